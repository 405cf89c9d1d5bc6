// Shared-memory ring for the row-streaming conversions: one producer thread
// moves groups of whole rows from global memory into a ring of stages with
// bulk asynchronous copies (cp.async.bulk, completion counted in bytes on the
// stage's "full" mbarrier); the consumer warps convert from shared memory and
// store their results straight to global memory, then release the stage on its
// "empty" mbarrier.  The copies keep kStages stages of input in flight per CTA
// whatever the consumers' register use, so the loads no longer wait behind the
// conversion arithmetic.
//
// The groups may also be 2D tiles moved by TMA tensor copies (the column-wise
// quantizers): `encode_bf16_tile_map` builds their tensor maps.
//
// Every wait is bounded.  A wait that runs out sets a bit in the library's
// status word and an abort flag the other roles poll; the producer then waits
// (bounded by time only) for the copies it has already issued before the CTA
// exits.  A stage is re-armed only after all consumer warps released it, so
// no barrier is re-armed with a transfer outstanding.
#pragma once

#include "common.cuh"
#include "tc.cuh"

namespace fp4q {
namespace ring {

constexpr int kStages = 4;                             // default ring depth
constexpr int kMaxStages = 8;
constexpr int kMaxConsumerWarps = 8;
constexpr int kMaxThreads = 32 * (1 + kMaxConsumerWarps);
constexpr uint32_t kHeaderBytes = 256;                 // barriers (2 x kMaxStages) + abort flag
constexpr uint64_t kWaitLimitNs = 2000000000ull;       // 2 s
constexpr uint32_t kMaxStageBytes = 16384;

// Launch shape of a ring kernel over rows of `units` work items (one per
// consumer thread and step) and `row_bytes` staged bytes: rows per stage and
// consumer warps chosen so that the stage's items fill the consumer threads
// as evenly as possible (ties: more warps, fewer rows).  rps = 0 when one row
// does not fit a stage.
struct Shape { uint32_t rps, warps; };

inline Shape ring_shape(uint32_t units, uint32_t row_bytes) {
    Shape best{0, 0};
    if (units == 0 || row_bytes == 0 || row_bytes > kMaxStageBytes) return best;
    double best_eff = -1.0;
    for (uint32_t w = kMaxConsumerWarps; w >= 4; --w)
        for (uint32_t r = 1; r * row_bytes <= kMaxStageBytes; ++r) {
            const uint32_t n = r * units, t = 32 * w;
            const double eff = double(n) / double((n + t - 1) / t * t);
            if (eff > best_eff + 1e-9) { best_eff = eff; best = Shape{r, w}; }
        }
    return best;
}
inline uint32_t smem_bytes(uint32_t stage_bytes, int stages = kStages) {
    return kHeaderBytes + uint32_t(stages) * stage_bytes;
}

// Tensor map of a BF16 [rows, cols] matrix (row stride ld elements) for TMA
// tile loads of box_cols x box_rows elements, no swizzle (dense rows).
fp4q_status encode_bf16_tile_map(CUtensorMap* map, const void* x, int64_t rows, int64_t cols, int64_t ld,
                                 uint32_t box_cols, uint32_t box_rows);

struct Ring {
    uint8_t* stage0;          // first stage (128-byte aligned)
    uint32_t stage_bytes;
    int stages;
    uint32_t bar0;            // full[stages] then empty[stages]
    volatile int* abort;

    __device__ uint32_t full(int s) const { return bar0 + 8u * uint32_t(s); }
    __device__ uint32_t empty(int s) const { return bar0 + 8u * uint32_t(stages + s); }
    __device__ uint8_t* stage(int s) const { return stage0 + uint32_t(s) * stage_bytes; }
};

// Called by every thread of the CTA; thread 0 initialises the barriers.  The
// CTA is one producer warp and blockDim.x / 32 - 1 consumer warps.
__device__ __forceinline__ Ring make_ring(uint8_t* smem, uint32_t stage_bytes, int stages = kStages) {
    Ring r;
    r.stage0 = smem + kHeaderBytes;
    r.stage_bytes = stage_bytes;
    r.stages = stages;
    r.bar0 = tc::smem_u32(smem);
    r.abort = reinterpret_cast<volatile int*>(smem + 8 * 2 * kMaxStages);
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            tc::mbar_init(r.full(s), 1);
            tc::mbar_init(r.empty(s), blockDim.x / 32 - 1);
        }
        *r.abort = 0;
        tc::fence_barrier_init();
    }
    __syncthreads();
    return r;
}

__device__ __forceinline__ void flag_abort(const Ring& r, uint32_t* status, uint32_t bit) {
    if (!*r.abort) {
        *r.abort = 1;
        atomicOr(status, bit);
    }
}

// Producer loop (one thread).  `issue(stage_ptr, full_bar, group)` arms the
// full barrier with the stage's byte count and issues its copies.
template <typename Issue>
__device__ __forceinline__ void produce(const Ring& r, int64_t ngroups, uint32_t* status, uint32_t bit,
                                        Issue issue) {
    int stage = 0;
    uint32_t phase = 0;
    int64_t issued = 0;
    for (int64_t g = blockIdx.x; g < ngroups; g += gridDim.x) {
        if (!tc::mbar_wait(r.empty(stage), phase ^ 1, r.abort, kWaitLimitNs)) {
            flag_abort(r, status, bit);
            break;
        }
        issue(r.stage(stage), r.full(stage), g);
        ++issued;
        if (++stage == r.stages) { stage = 0; phase ^= 1; }
    }
    // the copies already issued land before the CTA may exit
    for (int64_t i = 0; i < r.stages && i < issued; ++i) {
        if (--stage < 0) { stage = r.stages - 1; phase ^= 1; }
        if (!tc::mbar_wait_drain(r.full(stage), phase, kWaitLimitNs)) {
            flag_abort(r, status, bit);
            break;
        }
    }
}

// Consumer loop (all lanes of each consumer warp).  `consume(stage_ptr, group)`
// converts one stage; the warp then releases it.  A warp stops as a whole when
// any of its lanes saw the wait give up.
template <typename Consume>
__device__ __forceinline__ void consume(const Ring& r, int64_t ngroups, uint32_t* status, uint32_t bit,
                                        Consume fn) {
    const int lane = threadIdx.x & 31;
    int stage = 0;
    uint32_t phase = 0;
    for (int64_t g = blockIdx.x; g < ngroups; g += gridDim.x) {
        const bool got = tc::mbar_wait(r.full(stage), phase, r.abort, kWaitLimitNs);
        if (!__all_sync(0xffffffffu, got)) {
            if (lane == 0) flag_abort(r, status, bit);
            break;
        }
        fn(r.stage(stage), g);
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(r.empty(stage));
        if (++stage == r.stages) { stage = 0; phase ^= 1; }
    }
}

// As consume, for consumers that synchronise among themselves inside `fn`
// (named barrier 2): the go / give-up decision is taken by all consumer
// threads together (a barrier AND-reduction on named barrier 1), so no warp
// can stop while another waits for it at barrier 2.
template <typename Consume>
__device__ __forceinline__ void consume_together(const Ring& r, int64_t ngroups, uint32_t* status, uint32_t bit,
                                                 Consume fn) {
    const uint32_t nthreads = blockDim.x - 32;
    int stage = 0;
    uint32_t phase = 0;
    for (int64_t g = blockIdx.x; g < ngroups; g += gridDim.x) {
        const bool got = tc::mbar_wait(r.full(stage), phase, r.abort, kWaitLimitNs);
        if (!tc::named_bar_and(1, nthreads, got)) {
            if (threadIdx.x == 32) flag_abort(r, status, bit);
            break;
        }
        fn(r.stage(stage), g);
        __syncwarp();
        if ((threadIdx.x & 31) == 0) tc::mbar_arrive(r.empty(stage));
        if (++stage == r.stages) { stage = 0; phase ^= 1; }
    }
}

}  // namespace ring
}  // namespace fp4q
