// Q1_0 x Q8_0 decode GEMV, grouped layer sweep and the persistent single-matrix launch on sm_103a
// (browseml-gpu.js, header comment and Q1_DOT_WGSL): the exact per-row order of the pages, with the
// integer lane sums formed by dp4a (q1_common.cuh states how).
#include "q1_common.cuh"

namespace gq {
namespace {

// --------------------------------------------------------------------------------------------
// Decode GEMV, in two launches.
//  1. act_prep_kernel builds each activation's constants once per call into the caller's
//     workspace (per 32-activation sub-block: 8 quant words, 8 seeds, 8 scales = 96 bytes) and
//     zeroes the unit counter.  The GEMV is launched as its programmatic dependent, so the GEMV's
//     thread blocks are set up while it runs.
//  2. q1_gemv_kernel: persistent warps.  A unit is a 128-row tile of one matrix (four rows per
//     lane: each activation word is loaded once for four rows); units are handed out through the
//     counter, largest matrix first, so the greedy hand-out balances the warps.  Each warp streams
//     its units' (unit, block) chunks -- the tile's sign bits and d0 of the block plus the
//     block's 384 bytes of constants -- through a private ring of kStages stages of two blocks
//     each (two consecutive blocks' chunks are contiguous, and so are their constants, so a stage
//     is still two bulk copies): lane 0 refills the stage it has just consumed with the blocks
//     kStages stages ahead, so the copies run ahead across unit boundaries, and the waits and
//     refills come once per two blocks.  Lane 0 claims the next unit when it requests the last block of the
//     current one, so the counter's round trip overlaps a block of work.  The unit of each chunk
//     run travels through a small per-warp queue; the end of the work is a full-barrier phase
//     completed without data.  Every wait is bounded, and a warp that gives up first lets its
//     copies in flight land.  A problem with fewer tiles than the grid has warps is spread over
//     as many SMs as it has tiles.
// --------------------------------------------------------------------------------------------
// Measured on GB300 over the BitNet-2B layer sweep: four rows per lane beats one or two rows per
// lane shared by four or two warps (more warps fit, but the per-row cost of the block constants
// grows faster than the latency hiding), and cutting the last tiles into block runs that hand
// their accumulators on (for an even finish) costs as much as the uneven finish it removes.
constexpr int kGemvR = 4;                                   // rows per lane: a warp covers a tile
constexpr int kGemvWarps = 16;                              // 4 per SMSP (124 registers each)
constexpr int kStages = 2;
constexpr int kStageBlocks = 2;                             // blocks per ring stage
constexpr int kCstBytes = 4 * kConstWords * 4;              // 384: constants of one block
constexpr int kTileBits = kTileRows * 16;                   // sign bits of one (tile, block)
constexpr int kTileD0 = kTileRows * 2;                      // d0 of one (tile, block)
constexpr int kStageBytes = kStageBlocks * (kTileBits + kTileD0 + kCstBytes);
constexpr int kCachedDescs = 2048;                          // tile_begin cached in smem up to this
constexpr int kUnitQueue = 16;                              // > kStages + 1: units requested ahead
static_assert(kUnitQueue > kStages + 1, "unit queue too short");

// Lane 0's cursor over the chunks still to request.
struct Fetcher {
    const uint8_t* base;   // current unit's tile, first chunk
    const uint8_t* cst;    // its matrix's constants
    int blk, blk_end;      // next block to request, blocks of the unit
    int qi, issued;        // queue slot of the next unit, chunks requested so far
    int live;
};

struct __align__(16) WarpSmem {
    uint8_t ring[kStages][kStageBytes];
    uint64_t full[kStages];
    int units[kUnitQueue];
    Fetcher f;
};

struct TileInfo {
    const uint8_t* base;   // first chunk of the tile
    const uint8_t* cst;    // the matrix's activation constants (workspace)
    float* y;
    int rows;              // rows of the matrix
    int nb;                // blocks per row
    int row0;              // first row of the tile
};

// Descriptor of tile `tile`: binary search of tile_begin (shared-memory copy when the group is
// small enough, else global), then one read of the descriptor.
__device__ __forceinline__ TileInfo tile_info(const gq_gemv_desc& single, const gq_gemv_desc* __restrict__ descs,
                                              int count, const int* s_tb, int tile) {
    gq_gemv_desc d;
    if (count == 0) {
        d = single;
    } else {
        int lo = 0, hi = count - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            const int tb = (count <= kCachedDescs) ? s_tb[mid] : descs[mid].tile_begin;
            if (tb <= tile) lo = mid;
            else hi = mid - 1;
        }
        d = descs[lo];
    }
    TileInfo t;
    const int lt = tile - d.tile_begin;
    t.nb = d.n / 128;
    t.base = static_cast<const uint8_t*>(d.packed_w) + static_cast<size_t>(lt) * t.nb * kChunkBytes;
    t.cst = static_cast<const uint8_t*>(d.workspace);
    t.y = d.y;
    t.rows = d.rows;
    t.row0 = lt * kTileRows;
    return t;
}

__global__ void __launch_bounds__(256)
act_prep_kernel(gq_gemv_desc single, const gq_gemv_desc* __restrict__ descs, int count, int* counter) {
    // launched as a programmatic dependent of the work before it on the stream (often the previous
    // GEMV, which still uses the workspace and the counter): everything is read and written after
    // this wait, and only the launch and the thread blocks' start overlap that work's end
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // the GEMV grid may launch now; its griddepcontrol.wait still waits for this grid's writes
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const gq_gemv_desc d = (count == 0) ? single : descs[blockIdx.y];
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *counter = 0;
    const int items = (d.n / 32) * 8;     // a multiple of 32: whole warps take part in every step
    const uint8_t* act = static_cast<const uint8_t*>(d.act);
    uint32_t* ws = static_cast<uint32_t*>(d.workspace);
    for (int it = blockIdx.x * blockDim.x + threadIdx.x; it < items; it += gridDim.x * blockDim.x) {
        const int kg = it >> 3, l = it & 7;
        uint32_t qt, seed;
        float d1s;
        if (d.act_format == GQ_ACT_F32)
            act_lane_consts_f32(static_cast<const float*>(d.act), kg, l, qt, seed, d1s);
        else
            act_lane_consts(reinterpret_cast<const uint16_t*>(act + static_cast<size_t>(kg) * 34), l, qt, seed, d1s);
        ws[kg * kConstWords + l] = qt;
        ws[kg * kConstWords + 8 + l] = seed;
        ws[kg * kConstWords + 16 + l] = __float_as_uint(d1s);
    }
}

struct GemvArgs {
    gq_gemv_desc single;
    const gq_gemv_desc* descs;
    int count;
    int total_tiles;
    int active_warps;      // warps per thread block that take part
    int* counter;
};

// Lane 0: request the next chunk of the warp's stream into stage `s` (or, once the units have
// run out, complete that stage's next phase without data after posting -1).
// next_unit is lane 0's register holding the unit claimed when the current unit's last block was
// requested (its round trip overlaps a block of work).
__device__ __forceinline__ void fetch_next(WarpSmem& ws, int& next_unit, int s, const GemvArgs& a,
                                           const int* s_tb) {
    Fetcher& F = ws.f;
    if (!F.live) return;
    if (F.blk == F.blk_end) {                  // current unit fully requested: start the next one
        const int unit = next_unit;
        if (unit >= a.total_tiles) {
            ws.units[F.qi % kUnitQueue] = -1;
            mbar_arrive(&ws.full[s]);
            ++F.issued;
            F.live = 0;
            return;
        }
        ws.units[F.qi % kUnitQueue] = unit;
        ++F.qi;
        const TileInfo t = tile_info(a.single, a.descs, a.count, s_tb, unit);
        F.base = t.base;
        F.cst = t.cst;
        F.blk = 0;
        F.blk_end = t.nb;
    }
    // up to kStageBlocks consecutive blocks of the unit: their chunks are contiguous, and so are
    // their constants
    const int nblk = min(kStageBlocks, F.blk_end - F.blk);
    const uint8_t* ch = F.base + static_cast<size_t>(F.blk) * kChunkBytes;
    mbar_arrive_expect_tx(&ws.full[s], static_cast<uint32_t>(nblk) * (kTileBits + kTileD0 + kCstBytes));
    bulk_g2s(ws.ring[s], ch, nblk * (kTileBits + kTileD0), &ws.full[s]);
    bulk_g2s(ws.ring[s] + kStageBlocks * (kTileBits + kTileD0), F.cst + static_cast<size_t>(F.blk) * kCstBytes,
             nblk * kCstBytes, &ws.full[s]);
    F.blk += nblk;
    ++F.issued;
    if (F.blk == F.blk_end) next_unit = atomicAdd(a.counter, 1);     // consumed one block later
}

// Waits (bounded) for chunk c of the warp's stream.  After a timeout lane 0 lets the copies still
// in flight land before the warp's shared memory can be released.
__device__ __forceinline__ bool wait_chunk(WarpSmem& ws, int c, int lane) {
    const bool ok = __all_sync(0xffffffffu, mbar_wait(&ws.full[c % kStages], static_cast<uint32_t>(c / kStages) & 1u));
    if (!ok && lane == 0) {
        report_error(kErrWaitTimeout);
        for (int cc = c + 1; cc < ws.f.issued; ++cc)
            if (!mbar_wait(&ws.full[cc % kStages], static_cast<uint32_t>(cc / kStages) & 1u))
                report_error(kErrDrainTimeout);
    }
    return ok;
}

__global__ void __launch_bounds__(kGemvWarps * 32, 1)
q1_gemv_kernel(GemvArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    WarpSmem& ws = reinterpret_cast<WarpSmem*>(smem)[warp];
    int* s_tb = reinterpret_cast<int*>(smem + sizeof(WarpSmem) * kGemvWarps);
    if (a.count > 0 && a.count <= kCachedDescs)
        for (int i = threadIdx.x; i < a.count; i += blockDim.x) s_tb[i] = a.descs[i].tile_begin;
    const bool active = warp < a.active_warps;
    if (active && lane == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&ws.full[s], 1);
        fence_barrier_init();
    }
    __syncthreads();
    // launched as a programmatic dependent of act_prep_kernel: its constants and the zeroed unit
    // counter are visible after this wait (a no-op when launched the ordinary way)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // the next call's constants launch may start; it waits for this whole grid before it reads or
    // writes anything
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (!active) return;
    int next_unit = 0;
    if (lane == 0) {
        ws.f = Fetcher{nullptr, nullptr, 0, 0, 0, 0, 1};
        next_unit = atomicAdd(a.counter, 1);
        for (int s = 0; s < kStages; ++s) fetch_next(ws, next_unit, s, a, s_tb);
    }
    __syncwarp();

    int chunk = 0;
    for (int i = 0;; ++i) {
        if (!wait_chunk(ws, chunk, lane)) return;        // the unit's first chunk, or the end marker
        const int unit = ws.units[i % kUnitQueue];
        if (unit < 0) break;
        const TileInfo t = tile_info(a.single, a.descs, a.count, s_tb, unit);

        float2 acc[kGemvR][4];
#pragma unroll
        for (int j = 0; j < kGemvR; ++j)
#pragma unroll
            for (int p = 0; p < 4; ++p) acc[j][p] = make_float2(0.0f, 0.0f);

        for (int blk0 = 0; blk0 < t.nb; blk0 += kStageBlocks, ++chunk) {
            const int s = chunk % kStages;
            if (blk0 > 0 && !wait_chunk(ws, chunk, lane)) return;
            const int nblk = min(kStageBlocks, t.nb - blk0);
            const uint8_t* ring_s = ws.ring[s];
#pragma unroll
          for (int bb = 0; bb < kStageBlocks; ++bb) {   // the stage's blocks, in order
            if (bb >= nblk) break;                      // (unrolled: the offsets are constants)
            const uint8_t* stage = ring_s + bb * (kTileBits + kTileD0);
            uint4 wb[kGemvR];
            float d0[kGemvR];
#pragma unroll
            for (int j = 0; j < kGemvR; ++j) {
                wb[j] = reinterpret_cast<const uint4*>(stage)[lane + 32 * j];
                d0[j] = f16_to_f32(reinterpret_cast<const uint16_t*>(stage + kTileBits)[lane + 32 * j]);
            }
            const uint4* cst = reinterpret_cast<const uint4*>(ring_s + kStageBlocks * (kTileBits + kTileD0) +
                                                              bb * kCstBytes);

            float2 ab[kGemvR][4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint4* cs4 = cst + 6 * k;
                const uint4 q0 = cs4[0], q1 = cs4[1], s0 = cs4[2], s1 = cs4[3];
                const uint4 dd0 = cs4[4], dd1 = cs4[5];
                const float2 D01 = make_float2(__uint_as_float(dd0.x), __uint_as_float(dd0.y));
                const float2 D23 = make_float2(__uint_as_float(dd0.z), __uint_as_float(dd0.w));
                const float2 D45 = make_float2(__uint_as_float(dd1.x), __uint_as_float(dd1.y));
                const float2 D67 = make_float2(__uint_as_float(dd1.z), __uint_as_float(dd1.w));
                // k = 0: ab = D * (F - 1.5*2^23) as one fma, fma(D, F, -(D * 1.5*2^23)): D has at most
                // 11 significant bits, so -(D * 1.5*2^23) is exact, and the fma returns the exact
                // D * t (only an exact zero may come out as +0 instead of -0, which no later add can
                // carry into y, since acc starts at +0).  The four constants serve all rows.
                float2 N01, N23, N45, N67;
                if (k == 0) {
                    const float2 nm = make_float2(-kMagic, -kMagic);
                    N01 = fmul2(D01, nm);
                    N23 = fmul2(D23, nm);
                    N45 = fmul2(D45, nm);
                    N67 = fmul2(D67, nm);
                }
#pragma unroll
                for (int j = 0; j < kGemvR; ++j) {
                    const uint32_t w = (k == 0) ? wb[j].x : (k == 1) ? wb[j].y : (k == 2) ? wb[j].z : wb[j].w;
                    float2 tv[4];
                    if (k == 0) {
                        lane_words(w, q0, q1, s0, s1, tv);
                        ab[j][0] = ffma2(D01, tv[0], N01);
                        ab[j][1] = ffma2(D23, tv[1], N23);
                        ab[j][2] = ffma2(D45, tv[2], N45);
                        ab[j][3] = ffma2(D67, tv[3], N67);
                    } else {
                        lane_values(w, q0, q1, s0, s1, tv);
                        ab[j][0] = ffma2(D01, tv[0], ab[j][0]);
                        ab[j][1] = ffma2(D23, tv[1], ab[j][1]);
                        ab[j][2] = ffma2(D45, tv[2], ab[j][2]);
                        ab[j][3] = ffma2(D67, tv[3], ab[j][3]);
                    }
                }
            }
            if (bb == nblk - 1) {
                __syncwarp();                     // every lane has read the stage
                if (lane == 0) {
                    fence_proxy_async_smem();
                    fetch_next(ws, next_unit, s, a, s_tb);
                }
            }
#pragma unroll
            for (int j = 0; j < kGemvR; ++j) {
                const float2 dd = make_float2(d0[j], d0[j]);
#pragma unroll
                for (int p = 0; p < 4; ++p) acc[j][p] = ffma2(dd, ab[j][p], acc[j][p]);
            }
          }
        }
#pragma unroll
        for (int j = 0; j < kGemvR; ++j) {
            const int row = t.row0 + lane + 32 * j;
            if (row < t.rows) t.y[row] = final_reduce(acc[j]);
        }
    }
    // the end marker was the last phase requested: nothing is in flight
}

constexpr size_t kGemvSmem = sizeof(WarpSmem) * kGemvWarps + kCachedDescs * sizeof(int);

}  // namespace

GQ_ERROR_ACCESSOR(q1_gemv)

// Persistent grid (at most one thread block per SM and resident slot, cached per device).  A
// problem with fewer tiles than warps in a full grid is spread out: one thread block per tile up
// to the SM count, with only as many warps per block taking part as the tiles need.
static cudaError_t gemv_grid(int total_tiles, int* grid, int* active_warps) {
    static int cached[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (cached[dev] == 0) {
        e = cudaFuncSetAttribute(q1_gemv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kGemvSmem));
        if (e != cudaSuccess) return e;
        int sms = 0, per_sm = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, q1_gemv_kernel, kGemvWarps * 32, kGemvSmem);
        if (e != cudaSuccess) return e;
        cached[dev] = sms * (per_sm > 0 ? per_sm : 1);
    }
    const int g = total_tiles < cached[dev] ? total_tiles : cached[dev];
    int act = (total_tiles + g - 1) / g;
    if (act > kGemvWarps) act = kGemvWarps;
    *grid = g;
    *active_warps = act;
    return cudaSuccess;
}

// act_prep_kernel as a programmatic dependent of the work before it on `s` (see the kernel).
static cudaError_t launch_act_prep(int count, cudaStream_t s, const gq_gemv_desc& single,
                                   const gq_gemv_desc* descs, int* counter) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(8, count > 0 ? count : 1);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, act_prep_kernel, single, descs, count, counter);
}

// The GEMV grid as a programmatic dependent launch of the act_prep_kernel just queued on `s`: its
// thread blocks start (shared memory set-up, descriptor cache) while act_prep_kernel still runs.
static cudaError_t launch_gemv_dependent(int grid, cudaStream_t s, const GemvArgs& args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kGemvWarps * 32);
    cfg.dynamicSmemBytes = kGemvSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, q1_gemv_kernel, args);
}

// The activation constants, then 16 bytes for the tile counter.
size_t gemv_workspace_bytes(int n) { return static_cast<size_t>(n / 32) * kConstWords * 4 + 16; }

cudaError_t launch_q1_gemv_persistent(const void* packed, const void* act, float* y, int rows, int n,
                                      void* workspace, int act_format, cudaStream_t s) {
    const int tiles = gemv_tiles_for(rows);
    int grid = 0, active = 0;
    cudaError_t e = gemv_grid(tiles, &grid, &active);
    if (e != cudaSuccess) return e;
    int* counter = reinterpret_cast<int*>(static_cast<uint8_t*>(workspace) + gemv_workspace_bytes(n) - 16);
    gq_gemv_desc d{packed, act, y, workspace, rows, n, 0, act_format};
    e = launch_act_prep(0, s, d, nullptr, counter);
    if (e != cudaSuccess) return e;
    return launch_gemv_dependent(grid, s, GemvArgs{d, nullptr, 0, tiles, active, counter});
}

cudaError_t launch_q1_gemv_grouped(const gq_gemv_desc* descs, int count, int total_tiles, int* counter,
                                   cudaStream_t s) {
    int grid = 0, active = 0;
    cudaError_t e = gemv_grid(total_tiles, &grid, &active);
    if (e != cudaSuccess) return e;
    gq_gemv_desc none{nullptr, nullptr, nullptr, nullptr, 0, 128, 0, 0};
    e = launch_act_prep(count, s, none, descs, counter);
    if (e != cudaSuccess) return e;
    return launch_gemv_dependent(grid, s, GemvArgs{none, descs, count, total_tiles, active, counter});
}

}  // namespace gq
