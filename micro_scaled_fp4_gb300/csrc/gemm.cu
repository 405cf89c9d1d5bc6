// Block-scaled FP4 GEMMs on the sm_103a tensor cores: dense D = A . B^T and
// the grouped (per-expert, ragged) form of the MoE expert FFN.
//
// "Pretraining large language models with MXFP4 on Native FP4 Hardware",
// investigation section: the forward GEMM of a linear layer Y = X W^T with
// both operands in FP4 along the reduction axis, run on native FP4 tensor
// cores.  "Pretraining Large Language Models with NVFP4", section 2: NVFP4
// operands (E4M3 scale per 16, FP32 tensor scale); a Hadamard rotation of
// both operands along K cancels in the product.  "Practical FP4 Training for
// Large-Scale MoE Models on Hopper GPUs", section 2: MoE expert GEMMs over
// ragged per-expert row groups located by precomputed offsets, no padding.
//
// Persistent, warp-specialised kernel, one CTA per SM, 128 x 256 output tile
// per step, K consumed 256 elements (128 bytes) per pipeline stage:
//   warp 0      TMA producer: A and B tiles (128-byte swizzle; B as two
//               128-row halves) and the stage's block scales (contiguous
//               chunks of the MMA scale layout) into a ring of 3 to 6 stages;
//               the scales go first and land on their own barrier.
//   warp 1      allocates TMEM; one thread issues tcgen05.mma kind::mxf4
//               (UE8M0 per 32) or kind::mxf4nvf4 (UE4M3 per 16), FP32
//               accumulator in TMEM, reading the stage's block scales from
//               that stage's own TMEM scale buffer, once the stage's operands
//               have landed and its scales have been copied.
//   warps 10-11 one thread each copies half of each stage's block scales into
//               the stage's TMEM scale buffer (tcgen05.cp) as soon as they
//               have landed, while the operands still land; the two commits
//               release the scales to the MMA thread.  Issued from the MMA
//               thread, the copies held back the MMAs (a stage of MXFP4 took
//               ~830 cycles of issue for ~530 of MMA); from their own threads,
//               into buffers no MMA in flight reads, they overlap with the
//               MMAs.  The copy unit takes about 60 cycles per 512-byte chunk
//               (2 KB of TMEM once replicated to the four lane quadrants), so
//               an NVFP4 stage's 12 copies still exceed its 4 MMAs (~512).
//   warps 2..9  epilogue: tcgen05.ld of the 128 x 256 FP32 accumulator,
//               one row and half the columns per thread (two warps per TMEM
//               lane quadrant); the accumulator goes back to the MMA thread
//               as soon as it has been read (a relaxed arrive: it publishes
//               no memory).  STORE: scale, BF16
//               (round to nearest even) or FP32 stores.  SILU_GATE: the two
//               B halves are the gate and up rows of the same 128 outputs;
//               h = SiLU(gate) * up in FP32, then MXFP4 (one 32-element
//               block per 32 accumulator columns) straight from registers.
// Paired form (a cluster of two CTAs on two SMs, every tcgen05 instruction
// with .cta_group::2): the pair computes a 256 x 256 output tile with one MMA
// of M = 256 issued by the even CTA.  Each CTA loads its own 128 rows of A,
// its own 128-row half of the B tile and the block scales both of them need
// (its A rows, both B halves) into its own shared memory; its TMA loads count
// their bytes on the even CTA's "full" barrier, so the even CTA's MMA thread
// issues a stage once both CTAs have it, and its scale copies
// (tcgen05.cp .cta_group::2) fill each CTA's TMEM from that CTA's shared
// memory.  The even CTA's commits arrive on the "empty" and
// "accumulator full" barriers of both CTAs; each CTA's epilogue reads its own
// 128 TMEM lanes (its 128 output rows x 256 columns) and arrives, across the
// pair, on the even CTA's "accumulator empty" barrier.  Per SM this halves the
// B bytes a stage brings in and the MMA instructions per flop.  Dense MXFP4
// runs the paired form with six stages (see Layout), everything else paired
// with five; a dense GEMM of one 128-row tile runs the single-CTA form.
// Every mbarrier wait is bounded in time; a wait that gives up sets a bit in
// the library's status word and tells the other roles to stop.  The drain
// waits that follow (TMA loads issued, MMAs issued) do not stop on that flag,
// only on their own time limit, so the CTA frees TMEM and exits with no
// asynchronous work of its own in flight.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <string.h>

#include <atomic>
#include <type_traits>

#include "common.cuh"
#include "tc.cuh"

namespace fp4q {
namespace {

constexpr int BM = 128, BN = 256, BK = 256;           // elements
// Ring depth (single-CTA form): 3 stages, or 4 for MXFP8 operands, whose
// stages hold half the K of an FP4 stage and whose MMAs therefore wait on the
// loads more often.  With 3 stages the BF16 output goes through a
// shared-memory staging area and TMA stores; with 4 the staging area's room
// goes to the ring and the epilogue stores BF16 rows straight from registers.
// The paired form keeps 5 stages (6 for dense MXFP4) next to the staging.
constexpr uint32_t A_BYTES = BM * BK / 2;             // 16384
constexpr uint32_t B_HALF_BYTES = 128 * BK / 2;       // 16384
constexpr uint32_t B_BYTES = 2 * B_HALF_BYTES;
// BF16 output staging: two 64-column x 128-row boxes, rows of 128 bytes with the
// TMA 128-byte swizzle (16-byte chunk j of row r at chunk j ^ (r % 8)).
constexpr uint32_t BOX_BYTES = 128 * 128;             // 64 BF16 columns x 128 rows
// TMEM: FP32 accumulator in columns 0-255, then one block-scale buffer per
// ring stage (A: n chunks x 4 columns, B: 2 halves x n chunks x 4 columns,
// n = 4 or, in the six-stage layout, 2).
constexpr uint32_t TMEM_SF = 256;
// Per-CTA shared memory: NST ring stages [A | B (the pair: one half) | A
// scales | B scales], the BF16 staging boxes, barriers, the group prefix sums
// and the clamped group offsets.
//
// Six stages (paired, dense MXFP4 only): the ring is latency-bound -- a stage
// takes ~3400 cycles from its refill to its release, of which the landing from
// L2 is ~1650 -- so a sixth stage buys ~15 % on long K.  It fits by holding
// MXFP4's scales only (2 chunks of A and of each B half), one staging box, no
// group tables and 768 bytes of alignment slack (what is left of 227 KB):
// the kernel requires its dynamic shared memory to start within 768 bytes
// below a 1024-byte boundary (it starts on one, after the 1 KB the hardware
// reserves) and reports an error otherwise.
template <int NST, bool PAIR>
struct Layout {
    static constexpr bool mx_only = NST == 6;
    static constexpr uint32_t sf_chunks = mx_only ? 2 : 4;          // scale chunks per 128 rows a stage holds
    static constexpr uint32_t sfa_bytes = sf_chunks * 512;
    static constexpr uint32_t sfb_half_bytes = sf_chunks * 512;
    static constexpr uint32_t stage_bytes = A_BYTES + (PAIR ? B_HALF_BYTES : B_BYTES) + sfa_bytes + 2 * sfb_half_bytes;
    static constexpr uint32_t sfa_off = A_BYTES + (PAIR ? B_HALF_BYTES : B_BYTES);
    static constexpr uint32_t sfb_off = sfa_off + sfa_bytes;
    // TMEM columns per stage: A chunk c at 4 c, B half h chunk c at sfb_col + 8 c + 4 h
    static constexpr uint32_t sfb_col = 4 * sf_chunks;
    static constexpr uint32_t sf_cols = 3 * sfb_col;
    static constexpr uint32_t prefix_bytes = mx_only ? 0 : 12 * 260;   // tile, pair prefix sums, clamped offsets
    static constexpr uint32_t slack_max = 1024;
    static constexpr uint32_t nbox_max = mx_only ? 1 : 2;
    static constexpr bool staged_store =
        NST * stage_bytes + nbox_max * BOX_BYTES + 256 + prefix_bytes + (mx_only ? 0 : slack_max) <= 232448;
    static constexpr uint32_t nbox = staged_store ? nbox_max : 0;
    static constexpr uint32_t staging_bytes = nbox * BOX_BYTES;
    static constexpr uint32_t staging_off = NST * stage_bytes;
    static constexpr uint32_t bars_off = staging_off + staging_bytes;
    static constexpr uint32_t prefix_off = bars_off + 256;
    static constexpr uint32_t used_bytes = prefix_off + prefix_bytes;
    static constexpr uint32_t slack = used_bytes + slack_max <= 232448 ? slack_max : 232448 - used_bytes;
    static constexpr uint32_t smem_bytes = used_bytes + slack;
    static_assert(smem_bytes <= 232448, "GEMM shared memory above the 227 KB per-CTA limit");
    static_assert(4 * NST + 5 <= 30, "barriers overlap the TMEM slot");
    static_assert(TMEM_SF + sf_cols * NST <= 512, "scale buffers beyond the TMEM allocation");
    static_assert(!mx_only || (PAIR && staged_store), "the six-stage layout is the paired, staged one");
};
constexpr int kThreads = 384;          // producer warp, MMA warp, 8 epilogue warps, 2 scale-copy warps
constexpr uint32_t TMEM_COLS = 512;
constexpr uint64_t kWaitLimitNs = 4000000000ull;      // 4 s
constexpr int kMaxGroups = 256;            // the prefix / offset arrays hold kMaxGroups + 1 entries (260 reserved)
constexpr int kBandM = 32;                            // m-tiles per band of the dense tile order
constexpr int64_t kBandAboveBytes = 48ll << 20;       // band only an A operand L2 cannot keep

enum Epi { kStore = 0, kSiluGate = 1 };

struct GemmArgs {
    // dense: M rows of A, N rows of B.  grouped: rows of the dispatched A,
    // N rows of each group's B.
    int M, N, K;
    int n_tiles;                     // output tiles along N
    int k_stages;
    int nv;                          // 0 = MXFP4 / MXFP8 (UE8M0 / 32), 1 = NVFP4 (UE4M3 / 16)
    int f8;                          // 1 = MXFP8 operands (E4M3, one byte per element)
    int bk;                          // K elements per stage: 256 (FP4) or 128 (FP8); 128 bytes per row either way
    int groups;                      // 0 = dense
    int band_m;                      // dense: m-tiles per band of the tile order
    const int64_t* offsets;          // grouped: [groups + 1] row offsets
    const uint8_t* sfa;
    const uint8_t* sfb;
    uint64_t sf_tile_stride;         // bytes per 128-row tile of scales (A and B)
    uint32_t sf_box_bytes;           // paired form: bytes of one scale box (a stage's chunks of one 128-row tile)
    const float* ts_a;               // dense NVFP4: A tensor scale
    const float* ts_b;               // dense NVFP4: B tensor scale; grouped: [groups]
    const float* a_row_scale;        // grouped: per-row factor of A
    uint8_t* D;                      // STORE: [rows, ldd]; SILU_GATE: h codes [rows, N/4]
    int64_t ldd;                     // STORE: elements
    int d_bf16;
    uint8_t* h_scales;               // SILU_GATE: E8M0 [rows, N/64]
    float* h_debug;                  // SILU_GATE: optional FP32 h [rows, N/2]
    uint32_t* status;
    uint32_t status_bit;
};

struct TileInfo {
    int a_row0;       // first A row of the tile
    int row_end;      // rows >= row_end are not stored
    int a_sf_tile;    // 128-row scale tile of A
    int b_row0;       // first B row of each half (b_row1 < 0: half absent)
    int b_row1;
    int group;
    int col0;         // first output column
    bool phantom;     // paired form: this CTA's m-tile lies past the last one (loads for the pair, stores nothing)
};

__device__ __forceinline__ void flag_abort(volatile int* abort, uint32_t* status, uint32_t bit) {
    if (!*abort) {
        *abort = 1;
        atomicOr(status, bit);
    }
}

// Output tile `tile` -> rows / columns / scale tiles.  Grouped tiles run
// N-fastest, so the CTAs working at one time share A rows and one group's B.
// B rows of output-column tile nt of group `group` (both halves; b_row1 < 0:
// the second half lies past N).
template <int EPI>
__device__ __forceinline__ void decode_b(const GemmArgs& a, int nt, TileInfo& t) {
    const int gbase = t.group * a.N;
    if (EPI == kSiluGate) {
        t.b_row0 = gbase + nt * 128;
        t.b_row1 = gbase + a.N / 2 + nt * 128;
        t.col0 = nt * 128;
    } else {
        t.b_row0 = gbase + nt * BN;
        t.b_row1 = (nt * BN + 128 < a.N) ? t.b_row0 + 128 : -1;
        t.col0 = nt * BN;
    }
}

// Paired form: work unit `unit` -> this CTA's share (CTA rank `crank` of the
// pair takes m-tile 2 p + crank of the pair's m-tile pair p; both take the
// same B tile).  Grouped units pair the m-tiles of one group; dense units are
// banded over m-tile pairs like the single-CTA order.
template <int EPI>
__device__ __forceinline__ TileInfo decode_pair(const GemmArgs& a, int unit, const int* tile_prefix,
                                                const int* pair_prefix, const int* goff, int m_tiles,
                                                uint32_t crank) {
    TileInfo t;
    int nt, mp;
    if (a.groups) {
        nt = unit % a.n_tiles;
        mp = unit / a.n_tiles;
        int e = 0;
        while (e + 1 < a.groups && pair_prefix[e + 1] <= mp) ++e;
        const int lt = 2 * (mp - pair_prefix[e]) + int(crank);      // m-tile within the group
        const int tiles_e = tile_prefix[e + 1] - tile_prefix[e];
        t.group = e;
        t.phantom = lt >= tiles_e;
        t.a_row0 = goff[e] + lt * BM;
        t.row_end = goff[e + 1];
        t.a_sf_tile = tile_prefix[e] + min(lt, tiles_e - 1);
    } else {
        const int m_pairs = (m_tiles + 1) / 2, band_p = max(1, a.band_m / 2);
        const int band = unit / (band_p * a.n_tiles);
        const int within = unit - band * band_p * a.n_tiles;
        const int bs = min(band_p, m_pairs - band * band_p);
        nt = within / bs;
        mp = band * band_p + within % bs;
        const int mt = 2 * mp + int(crank);
        t.group = 0;
        t.phantom = mt >= m_tiles;
        t.a_row0 = mt * BM;
        t.row_end = a.M;
        t.a_sf_tile = min(mt, m_tiles - 1);
    }
    decode_b<EPI>(a, nt, t);
    return t;
}

template <int EPI>
__device__ __forceinline__ TileInfo decode_tile(const GemmArgs& a, int tile, const int* tile_prefix, const int* goff,
                                                int m_tiles) {
    TileInfo t;
    t.phantom = false;
    int nt, mt;
    if (a.groups) {
        nt = tile % a.n_tiles;
        mt = tile / a.n_tiles;
    } else {
        // dense: bands of band_m m-tiles; inside a band the m-tile runs fastest,
        // so the tiles in flight at once share one band of A (kept in L2 while
        // B streams past) instead of sweeping all of A every wave
        const int band = tile / (a.band_m * a.n_tiles);
        const int within = tile - band * a.band_m * a.n_tiles;
        const int bs = min(a.band_m, m_tiles - band * a.band_m);
        nt = within / bs;
        mt = band * a.band_m + within % bs;
    }
    if (a.groups) {
        int e = 0;
        while (e + 1 < a.groups && tile_prefix[e + 1] <= mt) ++e;
        const int local = mt - tile_prefix[e];
        t.group = e;
        t.a_row0 = goff[e] + local * BM;
        t.row_end = goff[e + 1];
    } else {
        t.group = 0;
        t.a_row0 = mt * BM;
        t.row_end = a.M;
    }
    t.a_sf_tile = mt;
    decode_b<EPI>(a, nt, t);
    return t;
}

// Converts 32 accumulator columns (FP32 bits) times alpha to 16 BF16 pairs.
__device__ __forceinline__ void to_bf16x32(const uint32_t (&r)[32], float alpha, uint32_t (&p)[16]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float lo = __fmul_rn(u2f(r[2 * i]), alpha), hi = __fmul_rn(u2f(r[2 * i + 1]), alpha);
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(p[i]) : "f"(hi), "f"(lo));
    }
}

// Writes 32 BF16 columns (chunk c of a 128-column half) of staging row `row`.
__device__ __forceinline__ void stage_bf16x32(uint32_t staging, int row, int c, const uint32_t (&p)[16]) {
    const uint32_t box = staging + uint32_t(c >> 1) * BOX_BYTES + uint32_t(row) * 128u;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t j = uint32_t((c & 1) * 4 + i);
        tc::st_shared_v4(box + ((j ^ uint32_t(row & 7)) << 4), p[4 * i], p[4 * i + 1], p[4 * i + 2], p[4 * i + 3]);
    }
}

// PAIR: launched as clusters of two CTAs (see the file comment); CG is the
// CTA group every tcgen05 instruction of the kernel names.
template <int EPI, int STAGES, bool PAIR>
__global__ void __launch_bounds__(kThreads, 1)
gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
            const __grid_constant__ CUtensorMap tmap_d, const __grid_constant__ CUtensorMap tmap_sfa,
            const __grid_constant__ CUtensorMap tmap_sfb, const GemmArgs args) {
    using LY = Layout<STAGES, PAIR>;
    constexpr int CG = PAIR ? 2 : 1;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    if constexpr (LY::slack < 1023) {
        // too little room to align every offset: every CTA of the launch sees the
        // same one and leaves
        if (uint32_t(smem - smem_raw) > LY::slack) {
            if (threadIdx.x == 0) atomicOr(args.status, args.status_bit);
            return;
        }
    }
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + LY::bars_off);
    // bars[0..STAGES) operands landed, [STAGES..2 STAGES) empty, then tmem_full,
    // tmem_empty, mma drain, [2 STAGES + 3 .. 3 STAGES + 3) scales copied, the two
    // copy threads' drains, [3 STAGES + 5 .. 4 STAGES + 5) scales landed
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 30);
    volatile int* abort = reinterpret_cast<volatile int*>(bars + 31);
    int* tile_prefix = reinterpret_cast<int*>(smem + LY::prefix_off);
    int* pair_prefix = tile_prefix + 260;
    int* goff = pair_prefix + 260;                  // the group offsets, clamped
    const uint32_t staging = tc::smem_u32(smem + LY::staging_off);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t bar0 = tc::smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto copied_bar = [&](int s) { return bar0 + 8u * (2 * STAGES + 3 + s); };
    auto sfull_bar = [&](int s) { return bar0 + 8u * (3 * STAGES + 5 + s); };
    const uint32_t tmem_full = bar0 + 8u * (2 * STAGES), tmem_empty = bar0 + 8u * (2 * STAGES + 1),
                   drain_bar = bar0 + 8u * (2 * STAGES + 2), cp_drain_bar = bar0 + 8u * (3 * STAGES + 3);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            tc::mbar_init(full_bar(s), 1);
            tc::mbar_init(empty_bar(s), 1);
            tc::mbar_init(copied_bar(s), 2);     // both copy threads' commits
            tc::mbar_init(sfull_bar(s), 1);
        }
        tc::mbar_init(tmem_full, 1);
        // one arrival per epilogue warp (the pair: the even CTA's barrier takes both CTAs' warps)
        tc::mbar_init(tmem_empty, PAIR ? 16 : 8);
        tc::mbar_init(drain_bar, 1);
        tc::mbar_init(cp_drain_bar, 1);
        tc::mbar_init(cp_drain_bar + 8, 1);
        *abort = 0;
        tc::fence_barrier_init();
        tc::tma_prefetch_desc(&tmap_a);
        tc::tma_prefetch_desc(&tmap_b);
        if constexpr (PAIR) {
            tc::tma_prefetch_desc(&tmap_sfa);
            tc::tma_prefetch_desc(&tmap_sfb);
        }
        // 128-row tiles per group and (paired form) pairs of them, prefix-summed.
        // Each offset is clamped into [previous offset, M] (the first into
        // [0, M]): well-formed offsets pass unchanged, and malformed ones can
        // make no tile read a row scale or store a row outside [0, M).
        if constexpr (!LY::mx_only) {
            int acc = 0, accp = 0, prev = 0;
            tile_prefix[0] = 0;
            pair_prefix[0] = 0;
            for (int e = 0; args.groups > 0 && e <= args.groups; ++e) {     // dense: no offsets
                const int o = int(min(max(args.offsets[e], int64_t(prev)), int64_t(args.M)));
                goff[e] = o;
                if (e > 0) {
                    const int tiles = (o - prev + BM - 1) / BM;      // group e - 1
                    acc += tiles;
                    accp += (tiles + 1) / 2;
                    tile_prefix[e] = acc;
                    pair_prefix[e] = accp;
                }
                prev = o;
            }
        }
    }
    if (warp == 1) {
        tc::tmem_alloc_g<CG>(tc::smem_u32(tmem_slot), TMEM_COLS);
        tc::tmem_relinquish_g<CG>();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t crank = PAIR ? tc::cluster_ctarank() : 0u;
    const bool leader = crank == 0;
    // the pair: both CTAs' barriers are initialised and their TMEM allocated
    if constexpr (PAIR) tc::cluster_sync_all();

    const int m_tiles = args.groups ? tile_prefix[args.groups] : (args.M + BM - 1) / BM;
    const int m_units = !PAIR ? m_tiles : (args.groups ? pair_prefix[args.groups] : (m_tiles + 1) / 2);
    const int num_tiles = m_units * args.n_tiles;
    const int unit0 = PAIR ? int(blockIdx.x >> 1) : int(blockIdx.x);
    const int unit_step = PAIR ? int(gridDim.x >> 1) : int(gridDim.x);
    const uint32_t chunk_elems = args.nv ? 64 : 128;  // K elements per 512-byte scale chunk
    auto decode = [&](int unit) {
        if constexpr (PAIR)
            return decode_pair<EPI>(args, unit, tile_prefix, pair_prefix, goff, m_tiles, crank);
        else
            return decode_tile<EPI>(args, unit, tile_prefix, goff, m_tiles);
    };

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer ----------------
        int stage = 0;
        uint32_t phase = 0;
        int issued = 0;
        bool ok = true;
        for (int tile = unit0; tile < num_tiles && ok; tile += unit_step) {
            const TileInfo t = decode(tile);
            for (int kb = 0; kb < args.k_stages; ++kb) {
                if (!tc::mbar_wait(empty_bar(stage), phase ^ 1, abort, kWaitLimitNs)) {
                    flag_abort(abort, args.status, args.status_bit);
                    ok = false;
                    break;
                }
                const int k_elems = min(args.bk, args.K - kb * args.bk);
                const uint32_t chunks = uint32_t(k_elems) / chunk_elems;
                const uint64_t ct0 = uint64_t(kb) * uint64_t(args.bk) / chunk_elems;
                const uint32_t sf_bytes = chunks * 512u * (t.b_row1 >= 0 ? 3u : 2u);
                uint8_t* st = smem + stage * LY::stage_bytes;
                const uint32_t fb = full_bar(stage);
                uint8_t* sfb_smem = st + LY::sfb_off;
                if constexpr (PAIR) {
                    // this CTA's A rows, B half `crank` and the scales of its A rows and
                    // of both B halves (an absent second half takes the first's scale
                    // tile: its columns are not stored); the bytes count on the even
                    // CTA's barriers, which expect both CTAs' boxes (every box lands in
                    // full, zero-filled where it leaves the tensor).  The scales go
                    // first and count on their own barrier: their copies to TMEM then
                    // overlap the operands' landing instead of following it.
                    const uint32_t fbp = tc::map_to_rank(fb, 0), sbp = tc::map_to_rank(sfull_bar(stage), 0);
                    if (leader) {
                        tc::mbar_arrive_expect_tx(sfull_bar(stage), 2u * 3u * args.sf_box_bytes);
                        tc::mbar_arrive_expect_tx(fb, 2u * (A_BYTES + B_HALF_BYTES));
                    }
                    const int brow = crank ? (t.b_row1 >= 0 ? t.b_row1 : t.b_row0 + 128) : t.b_row0;
                    const int bsf1 = (t.b_row1 >= 0 ? t.b_row1 : t.b_row0) / 128;
                    const uint64_t ck = ct0 * 512u;            // byte offset in a scale tile
                    tc::tma_load_2d_pair(tc::smem_u32(st + LY::sfa_off), &tmap_sfa, sbp, 0,
                                         int((uint64_t(t.a_sf_tile) * args.sf_tile_stride + ck) / 256u));
                    tc::tma_load_2d_pair(tc::smem_u32(sfb_smem), &tmap_sfb, sbp, 0,
                                         int((uint64_t(t.b_row0 / 128) * args.sf_tile_stride + ck) / 256u));
                    tc::tma_load_2d_pair(tc::smem_u32(sfb_smem + LY::sfb_half_bytes), &tmap_sfb, sbp, 0,
                                         int((uint64_t(bsf1) * args.sf_tile_stride + ck) / 256u));
                    tc::tma_load_2d_pair(tc::smem_u32(st), &tmap_a, fbp, kb * 128, t.a_row0);
                    tc::tma_load_2d_pair(tc::smem_u32(st + A_BYTES), &tmap_b, fbp, kb * 128, brow);
                } else {
                    // scales first, on their own barrier (as in the paired form)
                    const uint32_t sb = sfull_bar(stage);
                    tc::mbar_arrive_expect_tx(sb, sf_bytes);
                    tc::mbar_arrive_expect_tx(fb, A_BYTES + B_BYTES);
                    tc::bulk_load(tc::smem_u32(st + LY::sfa_off),
                                  args.sfa + uint64_t(t.a_sf_tile) * args.sf_tile_stride + ct0 * 512u, chunks * 512u,
                                  sb);
                    tc::bulk_load(tc::smem_u32(sfb_smem),
                                  args.sfb + uint64_t(t.b_row0 / 128) * args.sf_tile_stride + ct0 * 512u,
                                  chunks * 512u, sb);
                    if (t.b_row1 >= 0)
                        tc::bulk_load(tc::smem_u32(sfb_smem + LY::sfb_half_bytes),
                                      args.sfb + uint64_t(t.b_row1 / 128) * args.sf_tile_stride + ct0 * 512u,
                                      chunks * 512u, sb);
                    // x coordinate in bytes: 128 bytes of K per stage for both element widths
                    tc::tma_load_2d(tc::smem_u32(st), &tmap_a, fb, kb * 128, t.a_row0);
                    tc::tma_load_2d(tc::smem_u32(st + A_BYTES), &tmap_b, fb, kb * 128, t.b_row0);
                    // an absent second half still lands: rows past the end are zero-filled
                    tc::tma_load_2d(tc::smem_u32(st + A_BYTES + B_HALF_BYTES), &tmap_b, fb, kb * 128,
                                    t.b_row1 >= 0 ? t.b_row1 : t.b_row0 + 128);
                }
                ++issued;
                if (++stage == STAGES) { stage = 0; phase ^= 1; }
            }
        }
        // drain: every stage issued last must have landed before the CTA exits
        if (PAIR && !leader) {
            // the odd CTA's loads count on the even CTA's barriers: it waits for
            // the MMAs to have consumed its last fills (the data had landed)
            for (int i = max(0, issued - STAGES); i < issued; ++i) {
                if (!tc::mbar_wait_drain(empty_bar(i % STAGES), uint32_t(i / STAGES) & 1u, kWaitLimitNs)) {
                    flag_abort(abort, args.status, args.status_bit);
                    break;
                }
            }
        } else {
            for (int i = 0; i < STAGES && i < issued; ++i) {
                if (--stage < 0) { stage = STAGES - 1; phase ^= 1; }
                if (!tc::mbar_wait_drain(full_bar(stage), phase, kWaitLimitNs) ||
                    !tc::mbar_wait_drain(sfull_bar(stage), phase, kWaitLimitNs)) {
                    flag_abort(abort, args.status, args.status_bit);
                    break;
                }
            }
        }
    } else if (warp == 1 && lane == 0 && leader) {
        // ---------------- MMA issuer (the pair: the even CTA's) ----------------
        // Stage-0 descriptors, split into the low word (address field, advanced per
        // stage / K step) and the constant high word.  For the pair the same
        // shared-memory offsets address both CTAs' tiles.
        constexpr uint32_t MM = PAIR ? 2 * BM : BM;                 // rows of the MMA
        const uint64_t d0 = tc::smem_desc(tc::smem_u32(smem), 16, 1024, 2);
        const uint32_t d_lo0 = uint32_t(d0), d_hi = uint32_t(d0 >> 32);
        const uint32_t idesc_nv = tc::idesc_block_scaled(MM, BN, false, 0, 0);
        const uint32_t idesc_mx0 = tc::idesc_block_scaled(MM, BN, true, 0, 0);
        const uint32_t idesc_mx1 = tc::idesc_block_scaled(MM, BN, true, 2, 2);
        // MXFP8 (kind::mxf8f6f4, one UE8M0 byte per 32 elements): MMA j of a stage
        // reads byte j of the stage's scale column
        const uint32_t idesc_f8_0 = tc::idesc_block_scaled(MM, BN, true, 0, 0, 0, 0);
        const uint32_t idesc_f8_1 = tc::idesc_block_scaled(MM, BN, true, 1, 1, 0, 0);
        const uint32_t idesc_f8_2 = tc::idesc_block_scaled(MM, BN, true, 2, 2, 0, 0);
        const uint32_t idesc_f8_3 = tc::idesc_block_scaled(MM, BN, true, 3, 3, 0, 0);
        constexpr uint16_t kBoth = 0x3;                             // both CTAs of the pair
        int stage = 0;
        uint32_t phase = 0;
        int tcount = 0;
        bool ok = true;
        // This one thread's instruction stream paces the tensor pipe (a stage's
        // four MMAs take 512 cycles; with the operand format decided per stage the
        // thread needed ~700), so the loop is specialised per format: no format or
        // K-tail test inside a full stage.
        auto run = [&](auto fmt) {
            constexpr int F = decltype(fmt)::value;                  // 0 MXFP4, 1 NVFP4, 2 MXFP8
            // MMAs of stage `kb`: NM of them (K = 64 each for FP4, 32 for FP8)
            auto issue = [&](int kb, auto nm) {
                constexpr uint32_t NM = decltype(nm)::value;
                // descriptors of this stage: the 14-bit address field (bytes >> 4)
                // of the stage-0 descriptors advanced by the stage offset
                const uint32_t so = uint32_t(stage) * (LY::stage_bytes >> 4);
                const uint32_t a_lo = d_lo0 + so, b_lo = a_lo + (A_BYTES >> 4);
                // the stage's scale buffer: A chunk c at sfa + 4 c, B half h chunk c at sfb + 8 c + 4 h
                const uint32_t sfa = tmem + TMEM_SF + LY::sf_cols * uint32_t(stage), sfb = sfa + LY::sfb_col;
#pragma unroll
                for (uint32_t j = 0; j < NM; ++j) {
                    const uint64_t da = tc::desc_from(a_lo + 2 * j, d_hi), db = tc::desc_from(b_lo + 2 * j, d_hi);
                    const uint32_t acc = (kb | int(j)) ? 1u : 0u;
                    if constexpr (F == 2) {
                        // FP8: one scale chunk (A) and one per B half; MMA j reads byte j of each scale column
                        const uint32_t id = j == 0 ? idesc_f8_0 : j == 1 ? idesc_f8_1 : j == 2 ? idesc_f8_2 : idesc_f8_3;
                        tc::mma_mxf8_g<CG>(tmem, da, db, id, sfa, sfb, acc);
                    } else if constexpr (F == 1) {
                        // NVFP4: MMA j takes scale chunk j (4 x 16)
                        tc::mma_nvf4_g<CG>(tmem, da, db, idesc_nv, sfa + 4 * j, sfb + 8 * j, acc);
                    } else {
                        // MXFP4: MMA j takes half of chunk j / 2 (scale ids 0 / 2: its first or second pair)
                        tc::mma_mxf4_g<CG>(tmem, da, db, (j & 1) ? idesc_mx1 : idesc_mx0, sfa + 4 * (j >> 1),
                                           sfb + 8 * (j >> 1), acc);
                    }
                }
            };
            // The stage's operand tiles have landed (for the pair, both CTAs'
            // bytes) and the copy threads have put its scales in its TMEM buffer.
            // The two are separate barriers: the scales land first and their
            // copies overlap the operands' landing (with one barrier for both, a
            // stage went round the ring in ~3600 cycles, landing 1650 and copies
            // 780 of them; this thread has the time for a second wait).
            auto stage_ready = [&]() {
                if (!tc::mbar_wait(full_bar(stage), phase, abort, kWaitLimitNs) ||
                    !tc::mbar_wait(copied_bar(stage), phase, abort, kWaitLimitNs)) {
                    flag_abort(abort, args.status, args.status_bit);
                    ok = false;
                    return false;
                }
                tc::fence_after_sync();
                return true;
            };
            auto stage_done = [&]() {
                tc::tc_commit_g<CG>(empty_bar(stage), kBoth);     // the stage is free (in both CTAs)
                if (++stage == STAGES) { stage = 0; phase ^= 1; }
            };
            // FP4 stages hold 256 K elements; a K % 256 == 128 tail is one last
            // stage of two MMAs.  FP8 stages (128 elements) are always full.
            const int full = F == 2 ? args.k_stages : args.K / BK;
            for (int tile = unit0; tile < num_tiles && ok; tile += unit_step, ++tcount) {
                const bool got = PAIR ? tc::mbar_wait_cluster(tmem_empty, (tcount & 1) ^ 1, abort, kWaitLimitNs)
                                      : tc::mbar_wait(tmem_empty, (tcount & 1) ^ 1, abort, kWaitLimitNs);
                if (!got) {
                    flag_abort(abort, args.status, args.status_bit);
                    break;
                }
                tc::fence_after_sync();
                for (int kb = 0; kb < full; ++kb) {
                    if (!stage_ready()) break;
                    issue(kb, std::integral_constant<uint32_t, 4>{});
                    stage_done();
                }
                if (F != 2 && ok && full < args.k_stages) {
                    if (stage_ready()) {
                        issue(full, std::integral_constant<uint32_t, 2>{});
                        stage_done();
                    }
                }
                if (!ok) break;
                tc::tc_commit_g<CG>(tmem_full, kBoth);
            }
        };
        if (args.f8)
            run(std::integral_constant<int, 2>{});
        else if (args.nv)
            run(std::integral_constant<int, 1>{});
        else
            run(std::integral_constant<int, 0>{});
        // drain: all MMAs of this thread complete (a CTA that got no tile issued none)
        if (tcount > 0 || !ok) {
            tc::tc_commit_g<CG>(drain_bar, 0x1);
            if (!tc::mbar_wait_drain(drain_bar, 0, kWaitLimitNs)) flag_abort(abort, args.status, args.status_bit);
        }
    } else if (warp >= 10 && lane == 0 && leader) {
        // ---------------- scale copies (the pair: the even CTA's) ----------------
        // Per stage, once its scales have landed: the 512-byte scale chunks (128
        // rows x 4 scales) into the stage's TMEM buffer, replicated to the four
        // lane quadrants (for the pair, each CTA's chunks into its own TMEM) -- A
        // chunk c at column 4 c, B half h chunk c at 16 + 8 c + 4 h -- then a
        // commit on the stage's copied barrier, which the MMA thread waits for
        // besides the operands' barrier.  Copy thread `half` takes chunks
        // [half n / 2, (half + 1) n / 2) of the stage's n (one chunk: thread 0
        // the A chunk and B's first half, thread 1 B's second).
        // The buffer's previous contents were read by the MMAs of that stage's
        // previous fill, which completed before the stage was refilled.
        const uint32_t half = uint32_t(warp - 10);
        const uint64_t sf0 = tc::smem_desc(tc::smem_u32(smem + LY::sfa_off), 0, 128, 0);
        const uint32_t sf_lo0 = uint32_t(sf0), sf_hi = uint32_t(sf0 >> 32);
        int stage = 0;
        uint32_t phase = 0;
        int copied = 0;
        bool ok = true;
        for (int tile = unit0; tile < num_tiles && ok; tile += unit_step) {
            for (int kb = 0; kb < args.k_stages; ++kb) {
                if (!tc::mbar_wait(sfull_bar(stage), phase, abort, kWaitLimitNs)) {
                    flag_abort(abort, args.status, args.status_bit);
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                const uint32_t so = uint32_t(stage) * (LY::stage_bytes >> 4);
                const uint32_t sfa_lo = sf_lo0 + so, sfb_lo = sf_lo0 + so + (LY::sfa_bytes >> 4);
                const uint32_t sfa = tmem + TMEM_SF + LY::sf_cols * uint32_t(stage), sfb = sfa + LY::sfb_col;
                constexpr uint32_t h1 = LY::sfb_half_bytes >> 4;     // B's second half, in 16-byte units
                const uint32_t chunks = uint32_t(min(args.bk, args.K - kb * args.bk)) / chunk_elems;
                if (chunks == 4) {
#pragma unroll
                    for (uint32_t i = 0; i < 2; ++i) {
                        const uint32_t c = 2 * half + i;
                        tc::tc_cp_g<CG>(sfa + 4 * c, tc::desc_from(sfa_lo + 32 * c, sf_hi));
                        tc::tc_cp_g<CG>(sfb + 8 * c, tc::desc_from(sfb_lo + 32 * c, sf_hi));
                        tc::tc_cp_g<CG>(sfb + 8 * c + 4, tc::desc_from(sfb_lo + h1 + 32 * c, sf_hi));
                    }
                } else if (chunks == 2) {
                    const uint32_t c = half;
                    tc::tc_cp_g<CG>(sfa + 4 * c, tc::desc_from(sfa_lo + 32 * c, sf_hi));
                    tc::tc_cp_g<CG>(sfb + 8 * c, tc::desc_from(sfb_lo + 32 * c, sf_hi));
                    tc::tc_cp_g<CG>(sfb + 8 * c + 4, tc::desc_from(sfb_lo + h1 + 32 * c, sf_hi));
                } else if (half == 0) {
                    tc::tc_cp_g<CG>(sfa, tc::desc_from(sfa_lo, sf_hi));
                    tc::tc_cp_g<CG>(sfb, tc::desc_from(sfb_lo, sf_hi));
                } else {
                    tc::tc_cp_g<CG>(sfb + 4, tc::desc_from(sfb_lo + h1, sf_hi));
                }
                tc::tc_commit_g<CG>(copied_bar(stage), 0x1);
                ++copied;
                if (++stage == STAGES) { stage = 0; phase ^= 1; }
            }
        }
        // drain: the copies this thread issued complete before the CTA frees TMEM
        if (copied > 0) {
            tc::tc_commit_g<CG>(cp_drain_bar + 8 * half, 0x1);
            if (!tc::mbar_wait_drain(cp_drain_bar + 8 * half, 0, kWaitLimitNs))
                flag_abort(abort, args.status, args.status_bit);
        }
    } else if (warp >= 2 && warp < 10) {
        // ---------------- epilogue ----------------
        // Eight warps: warp w reads TMEM lane quadrant w % 4 (rows 32q .. 32q + 31 of
        // the tile) and the column half hf of the tile, so each warp's share of
        // the accumulator read (the part the MMA thread waits for) is 128 columns.
        const int q = warp & 3;
        const int hf = (warp - 2) >> 2;
        const int et = int(threadIdx.x) - 64;            // epilogue thread 0..255
        const float dense_alpha = (!args.groups && args.nv) ? __fmul_rn(*args.ts_a, *args.ts_b) : 1.0f;
        // the accumulator goes back to the MMA thread: one arrival per warp, on the
        // even CTA's barrier for the pair.  The arrival follows tcgen05.wait::ld
        // and publishes no memory, so it is relaxed.
        const uint32_t acc_empty = PAIR ? tc::map_to_rank(tmem_empty, 0) : tmem_empty;
        auto release_acc = [&]() {
            if constexpr (PAIR)
                tc::mbar_arrive_cluster_relaxed(acc_empty);
            else
                tc::mbar_arrive(acc_empty);
        };
        int tcount = 0;
        for (int tile = unit0; tile < num_tiles; tile += unit_step, ++tcount) {
            // The tile's coordinates and row factor come first, while the MMAs
            // still run: after the accumulator arrives they took ~650 cycles of
            // the hand-off in which the tensor pipe waits.
            const TileInfo t = decode(tile);
            const int row = t.a_row0 + q * 32 + lane;
            const bool row_ok = row < t.row_end;
            float alpha = dense_alpha;
            if (args.groups && row_ok) alpha = __fmul_rn(args.a_row_scale[row], args.ts_b[t.group]);
            const uint32_t lane_addr = tmem + (uint32_t(q * 32) << 16);
            // A warp that gives up on the accumulator flags the abort and still
            // runs the tile (its TMEM reads and stores are harmless; the call
            // reports the error), so that all eight warps meet at the staging
            // barriers; they decide together at the end of the tile whether to
            // stop.  (A vote here took ~190 cycles of the hand-off.)
            if (!tc::mbar_wait(tmem_full, tcount & 1, abort, kWaitLimitNs))
                flag_abort(abort, args.status, args.status_bit);
            tc::fence_after_sync();
            if constexpr (EPI == kSiluGate) {
                // h columns [64 hf, 64 hf + 64) of the tile: gate accumulator columns
                // 64 hf + j, up columns 128 + 64 hf + j
                const int hcols = args.N / 2;
                uint32_t g0[32], u0[32], g1[32], u1[32];
                tc::tmem_ld_32x32b_x32(lane_addr + uint32_t(64 * hf), g0);
                tc::tmem_ld_32x32b_x32(lane_addr + uint32_t(128 + 64 * hf), u0);
                tc::tmem_ld_32x32b_x32(lane_addr + uint32_t(64 * hf + 32), g1);
                tc::tmem_ld_32x32b_x32(lane_addr + uint32_t(128 + 64 * hf + 32), u1);
                tc::tmem_ld_wait();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) release_acc();
                if (row_ok) {
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const uint32_t(&g)[32] = c ? g1 : g0;
                        const uint32_t(&u)[32] = c ? u1 : u0;
                        float h[32];
                        uint32_t amax = 0;
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const float gv = __fmul_rn(u2f(g[i]), alpha);
                            const float uv = __fmul_rn(u2f(u[i]), alpha);
                            const float sig = __fdiv_rn(gv, __fadd_rn(1.0f, expf(-gv)));   // SiLU
                            h[i] = __fmul_rn(sig, uv);
                            amax = max(amax, f2u(h[i]) & 0x7fffffffu);
                        }
                        const int col = t.col0 + 64 * hf + 32 * c;
                        if (args.h_debug) {
                            float4* dbg = reinterpret_cast<float4*>(args.h_debug + int64_t(row) * hcols + col);
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                dbg[i] = make_float4(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
                        }
                        const int e = mx_exponent_from_amax_bits(amax);
                        const float inv = exp2i(-e);
                        uint32_t w[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            w[k] = cvt_e2m1x8(__fmul_rn(h[8 * k], inv), __fmul_rn(h[8 * k + 1], inv),
                                              __fmul_rn(h[8 * k + 2], inv), __fmul_rn(h[8 * k + 3], inv),
                                              __fmul_rn(h[8 * k + 4], inv), __fmul_rn(h[8 * k + 5], inv),
                                              __fmul_rn(h[8 * k + 6], inv), __fmul_rn(h[8 * k + 7], inv));
                        *reinterpret_cast<uint4*>(args.D + int64_t(row) * (hcols / 2) + col / 2) =
                            make_uint4(w[0], w[1], w[2], w[3]);
                        args.h_scales[int64_t(row) * (hcols / 32) + col / 32] = uint8_t(e + 127);
                    }
                }
            } else if (!LY::staged_store && args.d_bf16) {
                // BF16 from registers: the warp's 32 rows x 128 columns leave TMEM
                // first and the accumulator goes back to the MMA thread; then each
                // thread writes its row's 256 bytes with 16-byte stores.
                uint32_t hold[4][16];
#pragma unroll
                for (int c = 0; c < 4; c += 2) {
                    uint32_t r0[32], r1[32];
                    tc::tmem_ld_32x32b_x32(lane_addr + uint32_t(128 * hf + 32 * c), r0);
                    tc::tmem_ld_32x32b_x32(lane_addr + uint32_t(128 * hf + 32 * c + 32), r1);
                    tc::tmem_ld_wait();
                    to_bf16x32(r0, alpha, hold[c]);
                    to_bf16x32(r1, alpha, hold[c + 1]);
                }
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) release_acc();
                if (row_ok) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int col = t.col0 + 128 * hf + 32 * c;
                        uint8_t* dst = args.D + (int64_t(row) * args.ldd + col) * 2;
                        if (args.N - col >= 32) {
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                reinterpret_cast<uint4*>(dst)[i] =
                                    make_uint4(hold[c][4 * i], hold[c][4 * i + 1], hold[c][4 * i + 2], hold[c][4 * i + 3]);
                        } else if (col < args.N) {
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                if (i < args.N - col)
                                    reinterpret_cast<uint16_t*>(dst)[i] = uint16_t(hold[c][i >> 1] >> (16 * (i & 1)));
                        }
                    }
                }
            } else if (LY::staged_store && args.d_bf16 && !t.phantom &&
                       t.a_row0 + BM <= t.row_end + (args.groups ? 0 : BM)) {
                // BF16 through shared memory and TMA stores.  Each warp moves its 32 rows
                // x 128 columns out of TMEM into registers, then the accumulator goes
                // back to the MMA thread.  The tile leaves in four 64-column quarters
                // through the two staging boxes in turn: quarter q is staged while the
                // store of quarter q - 1 reads the other box (with whole 128-column
                // halves, staging waited for each half's store to have read the
                // staging: ~5500 cycles per tile, more than the MMAs of a K = 2048 tile).
                // The four loads go out together and the accumulator goes back before
                // any conversion: with the BF16 conversion between the loads, the read
                // phase took ~2500 cycles per tile, all of it idle tensor pipe.
                const int srow = q * 32 + lane;                  // row within the tile
                uint32_t raw[4][32];
#pragma unroll
                for (int c = 0; c < 4; ++c) tc::tmem_ld_32x32b_x32(lane_addr + uint32_t(128 * hf + 32 * c), raw[c]);
                tc::tmem_ld_wait();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) release_acc();
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) {
                    const int box = LY::nbox == 2 ? (qq & 1) : 0;
                    // the box's previous store (two quarters ago with two boxes, the
                    // last one with one; possibly the previous tile's) has read it
                    if (et == 0) {
                        if constexpr (LY::nbox == 2)
                            tc::bulk_wait_read1();
                        else
                            tc::bulk_wait_read0();
                    }
                    tc::named_bar_sync(1, 256);
                    if (hf == (qq >> 1)) {
#pragma unroll
                        for (int cc = 2 * (qq & 1); cc < 2 * (qq & 1) + 2; ++cc) {
                            uint32_t p[16];
                            to_bf16x32(raw[cc], alpha, p);
                            stage_bf16x32(staging, srow, LY::nbox == 2 ? cc : (cc & 1), p);
                        }
                    }
                    tc::fence_proxy_async_smem();
                    tc::named_bar_sync(1, 256);
                    if (et == 0) {
                        const int col = t.col0 + 64 * qq;
                        if (col < args.N) tc::tma_store_2d(&tmap_d, staging + uint32_t(box) * BOX_BYTES, col, t.a_row0);
                        tc::bulk_commit();
                    }
                }
            } else {
                // direct stores (FP32 output, or a tile that ends inside its group)
                for (int c = 0; c < 4; ++c) {
                    uint32_t r[32];
                    tc::tmem_ld_32x32b_x32(lane_addr + uint32_t(128 * hf + 32 * c), r);
                    tc::tmem_ld_wait();
                    if (c == 3) {
                        tc::fence_before_sync();
                        __syncwarp();
                        if (lane == 0) release_acc();
                    }
                    const int col = t.col0 + 128 * hf + c * 32;
                    if (!row_ok || col >= args.N) continue;
                    const int ncol = min(32, args.N - col);
                    if (args.d_bf16) {
                        uint32_t p[16];
                        to_bf16x32(r, alpha, p);
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
            if (!tc::named_bar_and(1, 256, *abort == 0)) break;
        }
    }
    if (EPI == kStore && threadIdx.x == 64) tc::bulk_wait0();   // the TMA stores this thread issued
    __syncwarp();          // the elected lanes rejoin their warps before the block barrier
    tc::fence_before_sync();
    __syncthreads();
    // the pair: neither CTA frees TMEM while the other may still read its
    // accumulator or arrive on its barriers
    if constexpr (PAIR) tc::cluster_sync_all();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc_g<CG>(tmem, TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
// Looked up on first use; concurrent first calls store the same pointer.
std::atomic<PFN_cuTensorMapEncodeTiled_v12000> g_encode_fn{nullptr};

fp4q_status get_encoder() {
    if (g_encode_fn.load(std::memory_order_acquire)) return FP4Q_OK;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
        return fail(FP4Q_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    g_encode_fn.store(reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn), std::memory_order_release);
    return FP4Q_OK;
}

// The encoder; valid once get_encoder() has returned FP4Q_OK.
PFN_cuTensorMapEncodeTiled_v12000 encoder() { return g_encode_fn.load(std::memory_order_acquire); }

// 2D map over operand bytes [rows, row_bytes] (K/2 for FP4, K for FP8):
// 128-byte x 128-row boxes, 128B swizzle.
fp4q_status encode_operand_map(CUtensorMap* map, const uint8_t* q, int64_t rows, int64_t row_bytes) {
    cuuint64_t dims[2] = {cuuint64_t(row_bytes), cuuint64_t(rows)};
    cuuint64_t strides[1] = {cuuint64_t(row_bytes)};
    cuuint32_t box[2] = {128u, 128u};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = encoder()(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(q), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(FP4Q_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", int(r));
    return FP4Q_OK;
}

// 2D map over a BF16 output [rows, ld] (N columns used): 64-column x 128-row
// boxes, 128B swizzle, for the TMA stores of the epilogue.
fp4q_status encode_output_map(CUtensorMap* map, void* D, int64_t rows, int64_t N, int64_t ld) {
    cuuint64_t dims[2] = {cuuint64_t(N), cuuint64_t(rows)};
    cuuint64_t strides[1] = {cuuint64_t(ld * 2)};
    cuuint32_t box[2] = {64u, 128u};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = encoder()(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(FP4Q_ERR_CUDA, "cuTensorMapEncodeTiled (output) failed (%d)", int(r));
    return FP4Q_OK;
}


// 2D map over a block-scale array in the MMA layout viewed as rows of 256
// bytes; a box is one stage's scale chunks of one 128-row tile (box_rows rows).
fp4q_status encode_scale_map(CUtensorMap* map, const uint8_t* s, uint64_t bytes, uint32_t box_rows) {
    cuuint64_t dims[2] = {256u, cuuint64_t(bytes / 256u)};
    cuuint64_t strides[1] = {256u};
    cuuint32_t box[2] = {256u, box_rows};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = encoder()(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(s), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(FP4Q_ERR_CUDA, "cuTensorMapEncodeTiled (scales) failed (%d)", int(r));
    return FP4Q_OK;
}

struct Maps {
    CUtensorMap a, b, d, sfa, sfb;
};

template <int EPI, int NST, bool PAIR>
fp4q_status launch_stages(const Maps& m, const GemmArgs& a, int units_upper, int sms, cudaStream_t stream) {
    constexpr uint32_t smem = Layout<NST, PAIR>::smem_bytes;
    auto kernel = gemm_kernel<EPI, NST, PAIR>;
    // per device, set on first use (setting it twice from racing threads is harmless)
    static std::atomic<bool> attr_set[64] = {};
    static std::atomic<int> max_clusters[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (!attr_set[dev & 63].load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e != cudaSuccess) return fail(FP4Q_ERR_CUDA, "gemm: smem attribute: %s", cudaGetErrorString(e));
        attr_set[dev & 63].store(true, std::memory_order_release);
    }
    if constexpr (PAIR) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        // pairs that fit on the GPU at once (one CTA per SM): the persistent grid
        int mc = max_clusters[dev & 63].load(std::memory_order_acquire);
        if (mc <= 0) {
            cfg.gridDim = dim3(unsigned(sms & ~1));
            const cudaError_t e = cudaOccupancyMaxActiveClusters(&mc, kernel, &cfg);
            if (e != cudaSuccess || mc <= 0) mc = sms / 2;
            max_clusters[dev & 63].store(mc, std::memory_order_release);
        }
        const int clusters = std::max(1, std::min(units_upper, mc));
        cfg.gridDim = dim3(unsigned(2 * clusters));
        const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, m.a, m.b, m.d, m.sfa, m.sfb, a);
        if (e != cudaSuccess) return fail(FP4Q_ERR_CUDA, "block_scaled_gemm (pair): %s", cudaGetErrorString(e));
        return FP4Q_OK;
    }
    const int grid = units_upper < sms ? units_upper : sms;
    kernel<<<grid, kThreads, smem, stream>>>(m.a, m.b, m.d, m.sfa, m.sfb, a);
    return check_launch("block_scaled_gemm");
}

// Ring depth: the paired form keeps 5 stages of 38 KB next to the BF16
// staging boxes, or, for dense MXFP4, 6 stages of 35 KB (see Layout); the
// single-CTA form 3 (FP4) or 4 (MXFP8, whose stages hold half the K of an FP4
// stage; its BF16 rows go out straight from registers).
constexpr int kPairStages = 5;
constexpr int kPairStagesMx = 6;

template <int EPI>
fp4q_status launch(const Maps& m, const GemmArgs& a, bool pair, int units_upper, int sms, cudaStream_t stream) {
    if (pair) {
        if constexpr (EPI == kStore) {
            if (!a.groups && !a.nv && !a.f8) return launch_stages<EPI, kPairStagesMx, true>(m, a, units_upper, sms, stream);
        }
        return launch_stages<EPI, kPairStages, true>(m, a, units_upper, sms, stream);
    }
    if constexpr (EPI == kStore) {
        if (a.f8) return launch_stages<EPI, 4, false>(m, a, units_upper, sms, stream);
    }
    return launch_stages<EPI, 3, false>(m, a, units_upper, sms, stream);
}

}  // namespace
}  // namespace fp4q

using namespace fp4q;

extern "C" fp4q_status fp4q_block_scaled_gemm(const fp4q_operand* A, const fp4q_operand* B, int64_t M,
                                              int64_t N, int64_t K, void* D, fp4q_dtype d_type, int64_t ldd,
                                              fp4q_stream_t stream) {
    if (!A || !B) return fail(FP4Q_ERR_INVALID_ARGUMENT, "gemm: operand is NULL");
    if (A->format != B->format || (A->format != FP4Q_MXFP4 && A->format != FP4Q_NVFP4 && A->format != FP4Q_MXFP8))
        return fail(FP4Q_ERR_INVALID_ARGUMENT, "gemm: A and B must have the same format (MXFP4, NVFP4 or MXFP8)");
    if (d_type != FP4Q_BF16 && d_type != FP4Q_FP32)
        return fail(FP4Q_ERR_INVALID_ARGUMENT, "gemm: d_type must be BF16 or FP32");
    if (M < 0 || N < 0 || K < 0 || ldd < N) return fail(FP4Q_ERR_INVALID_ARGUMENT, "gemm: bad sizes");
    if (K % 128) return fail(FP4Q_ERR_UNSUPPORTED_SHAPE, "gemm: K %% 128 != 0");
    if (M > (1 << 30) || N > (1 << 30) || K > (1 << 30))
        return fail(FP4Q_ERR_UNSUPPORTED_SHAPE, "gemm: sizes beyond 2^30");
    if (M == 0 || N == 0) return FP4Q_OK;
    if (((M + BM - 1) / BM) * ((N + BN - 1) / BN) > INT32_MAX)
        return fail(FP4Q_ERR_UNSUPPORTED_SHAPE, "gemm: more than 2^31 output tiles");
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
    Maps maps;
    memset(&maps, 0, sizeof maps);
    const bool f8 = A->format == FP4Q_MXFP8;
    const int64_t row_bytes = f8 ? K : K / 2;
    if ((st = encode_operand_map(&maps.a, A->q, M, row_bytes)) != FP4Q_OK) return st;
    if ((st = encode_operand_map(&maps.b, B->q, N, row_bytes)) != FP4Q_OK) return st;
    GemmArgs a = {};
    a.M = int(M);
    a.N = int(N);
    a.K = int(K);
    a.n_tiles = int((N + BN - 1) / BN);
    a.f8 = f8 ? 1 : 0;
    a.bk = f8 ? 128 : BK;
    a.k_stages = int((K + a.bk - 1) / a.bk);
    a.nv = nv ? 1 : 0;
    a.groups = 0;
    const int m_tiles = int((M + BM - 1) / BM);
    a.band_m = M * row_bytes > kBandAboveBytes ? std::min(kBandM, m_tiles) : m_tiles;
    a.sfa = A->scales;
    a.sfb = B->scales;
    a.sf_tile_stride = uint64_t(nv ? K / 64 : K / 128) * 512u;
    a.sf_box_bytes = uint32_t(a.bk / (nv ? 64 : 128)) * 512u;
    a.ts_a = A->tensor_scale;
    a.ts_b = B->tensor_scale;
    a.D = static_cast<uint8_t*>(D);
    a.ldd = ldd;
    a.d_bf16 = d_type == FP4Q_BF16;
    a.status = status_word();
    a.status_bit = kStatusGemmTimeout;
    if (a.d_bf16 && (st = encode_output_map(&maps.d, D, M, N, ldd)) != FP4Q_OK) return st;
    // paired CTAs whenever there are two m-tiles to pair
    const bool pair = m_tiles >= 2;
    if (pair) {
        const uint32_t box_rows = a.sf_box_bytes / 256u;
        if ((st = encode_scale_map(&maps.sfa, A->scales, uint64_t(m_tiles) * a.sf_tile_stride, box_rows)) != FP4Q_OK)
            return st;
        if ((st = encode_scale_map(&maps.sfb, B->scales, uint64_t((N + 127) / 128) * a.sf_tile_stride, box_rows)) !=
            FP4Q_OK)
            return st;
    }
    const int units = (pair ? (m_tiles + 1) / 2 : m_tiles) * a.n_tiles;
    return launch<kStore>(maps, a, pair, units, sms, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" fp4q_status fp4q_grouped_gemm(const uint8_t* a_q, const uint8_t* a_scales, const float* a_row_scale,
                                         const uint8_t* b_q, const uint8_t* b_scales, const float* b_tensor_scale,
                                         const int64_t* offsets, int64_t rows, int64_t groups, int64_t N, int64_t K,
                                         fp4q_epilogue epilogue, void* D, uint8_t* d_scales, float* h_debug,
                                         fp4q_stream_t stream) {
    if (epilogue != FP4Q_EPI_STORE_BF16 && epilogue != FP4Q_EPI_SILU_GATE_MXFP4)
        return fail(FP4Q_ERR_INVALID_ARGUMENT, "grouped_gemm: bad epilogue");
    if (rows < 0 || groups < 1 || groups > kMaxGroups || N < 1 || K < 0)
        return fail(FP4Q_ERR_INVALID_ARGUMENT, "grouped_gemm: need rows >= 0, 1 <= groups <= %d, N >= 1", kMaxGroups);
    if (K % 128) return fail(FP4Q_ERR_UNSUPPORTED_SHAPE, "grouped_gemm: K %% 128 != 0");
    if (N % 128) return fail(FP4Q_ERR_UNSUPPORTED_SHAPE, "grouped_gemm: N %% 128 != 0");
    if (epilogue == FP4Q_EPI_SILU_GATE_MXFP4 && N % 256)
        return fail(FP4Q_ERR_UNSUPPORTED_SHAPE, "grouped_gemm: gated epilogue needs N %% 256 == 0");
    if (rows > (1 << 30) || groups * N > (1 << 30) || K > (1 << 30))
        return fail(FP4Q_ERR_UNSUPPORTED_SHAPE, "grouped_gemm: sizes beyond 2^30");
    if (rows == 0) return FP4Q_OK;
    if (((rows + BM - 1) / BM + groups) * ((N + BN - 1) / BN) > INT32_MAX)
        return fail(FP4Q_ERR_UNSUPPORTED_SHAPE, "grouped_gemm: more than 2^31 output tiles");
    if (!a_q || !a_scales || !a_row_scale || !b_q || !b_scales || !b_tensor_scale || !offsets || !D ||
        (epilogue == FP4Q_EPI_SILU_GATE_MXFP4 && !d_scales))
        return fail(FP4Q_ERR_INVALID_ARGUMENT, "grouped_gemm: null pointer");
    if (!aligned16(a_q) || !aligned16(b_q) || !aligned16(a_scales) || !aligned16(b_scales) || !aligned16(D) ||
        (h_debug && !aligned16(h_debug)) || (reinterpret_cast<uintptr_t>(offsets) & 7u) ||
        (reinterpret_cast<uintptr_t>(a_row_scale) & 3u) || (reinterpret_cast<uintptr_t>(b_tensor_scale) & 3u))
        return fail(FP4Q_ERR_MISALIGNED, "grouped_gemm: operands and outputs must be 16-byte aligned");
    if (K == 0) return fail(FP4Q_ERR_UNSUPPORTED_SHAPE, "grouped_gemm: K == 0");
    int sms = 0;
    fp4q_status st = current_device(&sms);
    if (st != FP4Q_OK) return st;
    if ((st = get_encoder()) != FP4Q_OK) return st;
    Maps maps;
    memset(&maps, 0, sizeof maps);
    if ((st = encode_operand_map(&maps.a, a_q, rows, K / 2)) != FP4Q_OK) return st;
    if ((st = encode_operand_map(&maps.b, b_q, groups * N, K / 2)) != FP4Q_OK) return st;
    GemmArgs a = {};
    a.M = int(rows);
    a.N = int(N);
    a.K = int(K);
    a.bk = BK;
    a.k_stages = int((K + BK - 1) / BK);
    a.nv = 1;
    a.groups = int(groups);
    a.offsets = offsets;
    a.sfa = a_scales;
    a.sfb = b_scales;
    a.sf_tile_stride = uint64_t(K / 64) * 512u;
    a.sf_box_bytes = uint32_t(BK / 64) * 512u;
    a.ts_b = b_tensor_scale;
    a.a_row_scale = a_row_scale;
    a.D = static_cast<uint8_t*>(D);
    a.ldd = N;
    a.d_bf16 = 1;
    a.h_scales = d_scales;
    a.h_debug = h_debug;
    a.status = status_word();
    a.status_bit = kStatusGroupedTimeout;
    // the groups' m-tiles run as pairs (a group's odd last tile pairs with a
    // CTA that stores nothing): at most half the tiles plus one per group
    const int m_pairs_upper = int(((rows + BM - 1) / BM + groups) / 2 + groups);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const uint32_t box_rows = a.sf_box_bytes / 256u;
    const int m_tiles_upper = int((rows + BM - 1) / BM + groups);
    if ((st = encode_scale_map(&maps.sfa, a_scales, uint64_t(m_tiles_upper) * a.sf_tile_stride, box_rows)) != FP4Q_OK)
        return st;
    if ((st = encode_scale_map(&maps.sfb, b_scales, uint64_t(groups * N / 128) * a.sf_tile_stride, box_rows)) !=
        FP4Q_OK)
        return st;
    if (epilogue == FP4Q_EPI_SILU_GATE_MXFP4) {
        a.n_tiles = int(N / 256);
        return launch<kSiluGate>(maps, a, true, m_pairs_upper * a.n_tiles, sms, s);
    }
    if ((st = encode_output_map(&maps.d, D, rows, N, N)) != FP4Q_OK) return st;
    a.n_tiles = int((N + BN - 1) / BN);
    return launch<kStore>(maps, a, true, m_pairs_upper * a.n_tiles, sms, s);
}
