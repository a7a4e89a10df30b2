// Q1_0 weights x Q8_0 activations on sm_103a: one-time repack, decode GEMV (single matrix and
// grouped layer sweep) and the token-tiled GEMM (DP4A and LUT4 paths).
//
// Arithmetic (browseml-gpu.js, header comment and Q1_DOT_WGSL / Q1_MM_WGSL / Q1_MM4_WGSL): per
// row, per block i of 128 weights (f16 d0 + 128 sign bits), per sub-block k of 32 weights
// (Q8_0 block 4i+k: f16 d1 + 32 int8) and lane l (weights 4l..4l+3):
//   s = sum(bit ? q : -q) with the negate wrapping as int8;  p = d1*s (exact);
//   ab[l] = p (k = 0) or ab[l] + p;  acc[l] = fma(d0, ab[l], acc[l]);
//   y = ((a0+a4)+(a2+a6)) + ((a1+a5)+(a3+a7)).
//
// How the integer lane sums are formed here (the same values, fewer instructions):
//  * -128 quants: a -128 term is -128 whatever the bit, so with q~ = q except -128 -> 0 and
//    C = sum q~ + 128*count(-128),  s = 2*D - C  where D = sum over set bits of q~.
//  * The repack stores each 32-bit sign word bit-transposed: packed bit 8c+l = weight 4l+c.
//    Then (w & (0x01010101 << l)) holds lane l's four bits, one per byte, each worth 2^l, and
//    a single dp4a against the activation word l (bytes q~_{4l..4l+3}) gives 2^l * D.
//  * The dp4a accumulator starts at bits(1.5*2^23) - (sigma/2)*C, so its result read as f32 is
//    exactly 1.5*2^23 + (sigma/2)*s (sigma = 2^max(l,1), the lane's mask weight; lane 0's bits
//    are shifted up by one).  Subtracting 1.5*2^23 is exact, and multiplying by d1*2/sigma
//    gives exactly d1*s, so ab = fma(d1*2/sigma, t, ab) is the pages' rounded add.
//  * Pairs of lanes run through the packed f32x2 add/mul/fma (two IEEE operations each).
#include "gq_internal.cuh"

namespace gq {

namespace {

constexpr int kRPT = 4;          // rows per lane in the GEMV (a warp covers one 128-row tile)
constexpr uint32_t kMagicBits = 0x4B400000u;   // 1.5 * 2^23: ulp 1 in [2^23, 2^24)
constexpr float kMagic = 12582912.0f;
constexpr int kConstWords = 24;  // per 32-activation sub-block: 8 quant words, 8 seeds, 8 scales

// packed bit 8c + l <- page bit 4l + c (c = 0..3, l = 0..7)
__device__ __forceinline__ uint32_t transpose_signs(uint32_t w) {
    uint32_t out = 0;
#pragma unroll
    for (int l = 0; l < 8; ++l)
#pragma unroll
        for (int c = 0; c < 4; ++c) out |= ((w >> (4 * l + c)) & 1u) << (8 * c + l);
    return out;
}

__global__ void q1_pack_kernel(const uint8_t* __restrict__ raw, int rows, int nb,
                               uint8_t* __restrict__ packed, long long total) {
    long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= total) return;
    const int rr = static_cast<int>(idx % kTileRows);
    const long long tb = idx / kTileRows;          // tile * nb + block
    const int i = static_cast<int>(tb % nb);
    const long long tile = tb / nb;
    const long long row = tile * kTileRows + rr;
    uint8_t* chunk = packed + static_cast<size_t>(tb) * kChunkBytes;
    uint4 bits = make_uint4(0u, 0u, 0u, 0u);
    uint16_t d0 = 0;
    if (row < rows) {
        const uint8_t* b = raw + (static_cast<size_t>(row) * nb + i) * 18;
        d0 = static_cast<uint16_t>(b[0] | (b[1] << 8));
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            w[k] = static_cast<uint32_t>(b[2 + 4 * k]) | (static_cast<uint32_t>(b[3 + 4 * k]) << 8) |
                   (static_cast<uint32_t>(b[4 + 4 * k]) << 16) | (static_cast<uint32_t>(b[5 + 4 * k]) << 24);
        bits = make_uint4(transpose_signs(w[0]), transpose_signs(w[1]), transpose_signs(w[2]),
                          transpose_signs(w[3]));
    }
    reinterpret_cast<uint4*>(chunk)[rr] = bits;
    reinterpret_cast<uint16_t*>(chunk + kTileRows * 16)[rr] = d0;
}

// Activation constants of one (sub-block, lane l) from its f16 d1 bits and its four quants
// (little-endian word): the quant word with -128 zeroed, the dp4a seed and d1 * 2/sigma.
__device__ __forceinline__ void lane_consts(uint32_t d1bits, uint32_t qw, int l, uint32_t& qt, uint32_t& seed,
                                            float& d1s) {
    const float d1 = f16_to_f32(d1bits);
    int C = 0;
    uint32_t t = 0;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int q = static_cast<int>(static_cast<int8_t>((qw >> (8 * c)) & 0xFFu));
        if (q == -128) {
            C += 128;
        } else {
            C += q;
            t |= (static_cast<uint32_t>(q) & 0xFFu) << (8 * c);
        }
    }
    const int half_sigma = (l <= 1) ? 1 : (1 << (l - 1));
    qt = t;
    seed = kMagicBits - static_cast<uint32_t>(half_sigma * C);
    d1s = __fmul_rn(d1, 1.0f / static_cast<float>(half_sigma));   // power of two: exact
}

// The same from a 34-byte Q8_0 block in memory (2-byte aligned).
__device__ __forceinline__ void act_lane_consts(const uint16_t* blk, int l, uint32_t& qt, uint32_t& seed,
                                                float& d1s) {
    lane_consts(blk[0], static_cast<uint32_t>(blk[1 + 2 * l]) | (static_cast<uint32_t>(blk[2 + 2 * l]) << 16), l,
                qt, seed, d1s);
}

// The same from f32 activations, quantized to Q8_0 on the way (the values gq_quantize_q8_0 would
// store): lane l of sub-block kg quantizes x[32 kg + 4 l .. + 3] (v, already loaded); the
// sub-block's eight lanes are eight consecutive, 8-aligned lanes of the warp, which exchange their
// amax.
__device__ __forceinline__ void lane_consts_f32(const float4 v, int l, uint32_t& qt, uint32_t& seed, float& d1s) {
    float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float dd = q8_0_scale(amax);
    const uint32_t qw = (static_cast<uint32_t>(q8_0_quant(v.x, amax, dd)) & 0xFFu) |
                        ((static_cast<uint32_t>(q8_0_quant(v.y, amax, dd)) & 0xFFu) << 8) |
                        ((static_cast<uint32_t>(q8_0_quant(v.z, amax, dd)) & 0xFFu) << 16) |
                        (static_cast<uint32_t>(q8_0_quant(v.w, amax, dd)) << 24);
    lane_consts(__half_as_ushort(__float2half_rn(dd)), qw, l, qt, seed, d1s);
}
__device__ __forceinline__ void act_lane_consts_f32(const float* x, int kg, int l, uint32_t& qt, uint32_t& seed,
                                                    float& d1s) {
    lane_consts_f32(*reinterpret_cast<const float4*>(x + static_cast<size_t>(kg) * 32 + 4 * l), l, qt, seed, d1s);
}

// The eight dp4a results of one 32-weight sub-block word (transposed layout) read as f32, i.e.
// 1.5 * 2^23 + (sigma_l/2) * s_l, as four pairs (lanes 0-1, 2-3, 4-5, 6-7).
__device__ __forceinline__ void lane_words(uint32_t w, const uint4& q0, const uint4& q1, const uint4& s0,
                                           const uint4& s1, float2 f[4]) {
    const int r0 = dp4a_us(__funnelshift_l(0u, w, 1) & 0x02020202u, q0.x, static_cast<int>(s0.x));   // SHF: ALU pipe
    const int r1 = dp4a_us(w & 0x02020202u, q0.y, static_cast<int>(s0.y));
    const int r2 = dp4a_us(w & 0x04040404u, q0.z, static_cast<int>(s0.z));
    const int r3 = dp4a_us(w & 0x08080808u, q0.w, static_cast<int>(s0.w));
    const int r4 = dp4a_us(w & 0x10101010u, q1.x, static_cast<int>(s1.x));
    const int r5 = dp4a_us(w & 0x20202020u, q1.y, static_cast<int>(s1.y));
    const int r6 = dp4a_us(w & 0x40404040u, q1.z, static_cast<int>(s1.z));
    const int r7 = dp4a_us(w & 0x80808080u, q1.w, static_cast<int>(s1.w));
    f[0] = make_float2(__int_as_float(r0), __int_as_float(r1));
    f[1] = make_float2(__int_as_float(r2), __int_as_float(r3));
    f[2] = make_float2(__int_as_float(r4), __int_as_float(r5));
    f[3] = make_float2(__int_as_float(r6), __int_as_float(r7));
}

// The eight lane values t_l = (sigma_l/2) * s_l (the words minus 1.5 * 2^23, exactly).
__device__ __forceinline__ void lane_values(uint32_t w, const uint4& q0, const uint4& q1, const uint4& s0,
                                            const uint4& s1, float2 t[4]) {
    lane_words(w, q0, q1, s0, s1, t);
    const float2 nm = make_float2(-kMagic, -kMagic);
#pragma unroll
    for (int p = 0; p < 4; ++p) t[p] = fadd2(t[p], nm);
}

__device__ __forceinline__ float final_reduce(const float2 acc[4]) {
    // acc[0] = (a0,a1), acc[1] = (a2,a3), acc[2] = (a4,a5), acc[3] = (a6,a7)
    const float2 s0415 = fadd2(acc[0], acc[2]);     // (a0+a4, a1+a5)
    const float2 s2637 = fadd2(acc[1], acc[3]);     // (a2+a6, a3+a7)
    const float2 lohi = fadd2(s0415, s2637);        // ((a0+a4)+(a2+a6), (a1+a5)+(a3+a7))
    return __fadd_rn(lohi.x, lohi.y);
}

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

// --------------------------------------------------------------------------------------------
// Decode GEMV for a problem that leaves SMs idle (a single matrix with fewer 128-row tiles than
// the GPU has SMs): one launch, no workspace.  Only acc = fma(d0, ab, acc) runs in block order;
// the lane sums ab of different blocks are independent.  A thread block covers 32 rows: its
// kSmallWarps warps take the blocks in turn (warp w the blocks w, w + 16, ... of each group
// of 32 or 64), each lane one row; a warp builds its block's activation constants itself (one (sub-block, lane) item per
// lane), and leaves ab (two float4 per row: lane groups 0-3 and 4-7) and d0 in shared memory.
// Then warps 0 and 1 run the chains of lane groups 0-3 and 4-7 over the pass's blocks in order for
// the 32 rows, and at the end warp 0 adds each row's eight chains in the pages' order.  (Eight
// chain warps reading scalars cut one launch's latency no further and cost ~15% more instructions
// per thread block, which launches of several waves -- a few-token GEMM -- pay in full.)
// The kernel is launched as a programmatic dependent: it lets the next launch on the stream start
// at once, loads its first weights (which no preceding launch of this library writes) and only
// then waits for the preceding grids before it reads the activation or writes y.  In a stream of
// GEMVs (a decode step) the next matrix's weights are in flight while the current one finishes.
// --------------------------------------------------------------------------------------------
constexpr int kSmallWarps = 16;
constexpr int kSmallPass = 2 * kSmallWarps;   // blocks per pass through shared memory

// J: blocks per warp in a group (2 for rows of at most 32 blocks, which keeps the kernel within 64
// registers so that two thread blocks share an SM; 4 for longer rows)
template <int ACT, int J>   // ACT: GQ_ACT_Q8_0 or GQ_ACT_F32
__global__ void __launch_bounds__(kSmallWarps * 32)
q1_gemv_small_kernel(const uint8_t* __restrict__ packed, const uint8_t* __restrict__ act, float* __restrict__ y,
                     int rows, int nb) {
    __shared__ __align__(16) float4 s_ab[kSmallPass][2][32];            // ab of (block, row): two float4
    __shared__ float s_d0[kSmallPass][32];
    __shared__ __align__(16) uint32_t s_cst[kSmallWarps][4 * kConstWords];  // a warp's current block
    __shared__ float s_acc[8][32];                                      // the chains' results
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = blockIdx.x * 32;
    const int rq = row0 % kTileRows;                                     // rows within their tile
    // blockIdx.y: the column of a few-token GEMM (its activation and output row); 0 for a GEMV
    if (blockIdx.y > 0) {
        act += static_cast<size_t>(blockIdx.y) * nb * 4 * (ACT == GQ_ACT_F32 ? 128 : 34);
        y += static_cast<size_t>(blockIdx.y) * rows;
    }
    const uint8_t* tile_base = packed + static_cast<size_t>(row0 / kTileRows) * nb * kChunkBytes;
    // the cta's rows sit in a whole packed tile (packing pads the last tile), so every read below
    // stays inside the packed buffer; rows >= `rows` are computed and not stored
    float4 chain = make_float4(0.0f, 0.0f, 0.0f, 0.0f);   // warps 0, 1: lane groups 4w..4w+3 of row `lane`

    // groups of up to J * kSmallWarps blocks: warp w owns blocks w + 16 j (j < J) of a group, whose
    // sign words, d0 and activation items it loads up front; the group then goes through shared
    // memory in passes of 2 * kSmallWarps blocks
    constexpr int kGroupBlocks = J * kSmallWarps;
    for (int g0 = 0; g0 < nb; g0 += kGroupBlocks) {
        const int ng = min(kGroupBlocks, nb - g0);
        uint4 wbv[J];
        uint32_t d0b[J];
#pragma unroll
        for (int j = 0; j < J; ++j) {
            const int bl = warp + kSmallWarps * j;
            if (bl < ng) {
                const uint8_t* ch = tile_base + static_cast<size_t>(g0 + bl) * kChunkBytes;
                wbv[j] = *reinterpret_cast<const uint4*>(ch + (rq + lane) * 16);
                d0b[j] = *reinterpret_cast<const uint16_t*>(ch + kTileRows * 16 + (rq + lane) * 2);
            }
        }
        // the preceding grids' writes (the activation) are visible after this wait
        if (g0 == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
        // the activation items of the warp's blocks (lane 8k + l: sub-block k, lane l)
        const int k = lane >> 3, l = lane & 7;
        float4 xv[J];
        uint32_t d1raw[J], qwraw[J];
#pragma unroll
        for (int j = 0; j < J; ++j) {
            const int bl = warp + kSmallWarps * j;
            if (bl < ng) {
                const int kg = 4 * (g0 + bl) + k;
                if constexpr (ACT == GQ_ACT_F32) {
                    xv[j] = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(act) +
                                                             static_cast<size_t>(kg) * 32 + 4 * l);
                } else {
                    const uint16_t* blk = reinterpret_cast<const uint16_t*>(act + static_cast<size_t>(kg) * 34);
                    d1raw[j] = blk[0];
                    qwraw[j] = static_cast<uint32_t>(blk[1 + 2 * l]) | (static_cast<uint32_t>(blk[2 + 2 * l]) << 16);
                }
            }
        }
#pragma unroll
        for (int half = 0; half < J / 2; ++half) {
            const int p0 = half * kSmallPass;              // first block of the pass, within the group
            if (p0 >= ng) break;
            const int np = min(kSmallPass, ng - p0);
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                const int j = 2 * half + jj;
                const int bl = warp + kSmallWarps * jj;     // block of the pass
                if (bl >= np) break;
                {
                    uint32_t qt, seed;
                    float d1s;
                    if constexpr (ACT == GQ_ACT_F32)
                        lane_consts_f32(xv[j], l, qt, seed, d1s);
                    else
                        lane_consts(d1raw[j], qwraw[j], l, qt, seed, d1s);
                    s_cst[warp][k * kConstWords + l] = qt;
                    s_cst[warp][k * kConstWords + 8 + l] = seed;
                    s_cst[warp][k * kConstWords + 16 + l] = __float_as_uint(d1s);
                }
                __syncwarp();
                const uint4 wb = wbv[j];
                const uint4* cst = reinterpret_cast<const uint4*>(s_cst[warp]);
                float2 ab[4];
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint4* cs4 = cst + 6 * kk;
                    const uint4 q0 = cs4[0], q1 = cs4[1], s0 = cs4[2], s1 = cs4[3];
                    const uint4 dd0 = cs4[4], dd1 = cs4[5];
                    const float2 D01 = make_float2(__uint_as_float(dd0.x), __uint_as_float(dd0.y));
                    const float2 D23 = make_float2(__uint_as_float(dd0.z), __uint_as_float(dd0.w));
                    const float2 D45 = make_float2(__uint_as_float(dd1.x), __uint_as_float(dd1.y));
                    const float2 D67 = make_float2(__uint_as_float(dd1.z), __uint_as_float(dd1.w));
                    const uint32_t w = (kk == 0) ? wb.x : (kk == 1) ? wb.y : (kk == 2) ? wb.z : wb.w;
                    float2 tv[4];
                    lane_values(w, q0, q1, s0, s1, tv);
                    if (kk == 0) {
                        ab[0] = fmul2(D01, tv[0]);
                        ab[1] = fmul2(D23, tv[1]);
                        ab[2] = fmul2(D45, tv[2]);
                        ab[3] = fmul2(D67, tv[3]);
                    } else {
                        ab[0] = ffma2(D01, tv[0], ab[0]);
                        ab[1] = ffma2(D23, tv[1], ab[1]);
                        ab[2] = ffma2(D45, tv[2], ab[2]);
                        ab[3] = ffma2(D67, tv[3], ab[3]);
                    }
                }
                s_ab[bl][0][lane] = make_float4(ab[0].x, ab[0].y, ab[1].x, ab[1].y);
                s_ab[bl][1][lane] = make_float4(ab[2].x, ab[2].y, ab[3].x, ab[3].y);
                s_d0[bl][lane] = f16_to_f32(d0b[j]);
                __syncwarp();                      // the warp's constants are read before the next block
            }
            __syncthreads();
            if (warp < 2) {
#pragma unroll 4
                for (int bl = 0; bl < np; ++bl) {
                    const float d0 = s_d0[bl][lane];
                    const float4 v = s_ab[bl][warp][lane];
                    chain.x = __fmaf_rn(d0, v.x, chain.x);
                    chain.y = __fmaf_rn(d0, v.y, chain.y);
                    chain.z = __fmaf_rn(d0, v.z, chain.z);
                    chain.w = __fmaf_rn(d0, v.w, chain.w);
                }
            }
            __syncthreads();                       // the pass is consumed before the next overwrites it
        }
    }
    if (warp < 2) {
        s_acc[4 * warp][lane] = chain.x;
        s_acc[4 * warp + 1][lane] = chain.y;
        s_acc[4 * warp + 2][lane] = chain.z;
        s_acc[4 * warp + 3][lane] = chain.w;
    }
    __syncthreads();
    if (warp == 0) {
        const int row = row0 + lane;
        // ((a0 + a4) + (a2 + a6)) + ((a1 + a5) + (a3 + a7))
        const float lo = __fadd_rn(__fadd_rn(s_acc[0][lane], s_acc[4][lane]), __fadd_rn(s_acc[2][lane], s_acc[6][lane]));
        const float hi = __fadd_rn(__fadd_rn(s_acc[1][lane], s_acc[5][lane]), __fadd_rn(s_acc[3][lane], s_acc[7][lane]));
        if (row < rows) y[row] = __fadd_rn(lo, hi);
    }
}

// Launches `kernel` as a programmatic dependent of the work before it on `s` (the kernel itself
// waits with griddepcontrol.wait before it depends on that work).
template <typename... KArgs, typename... Args>
static cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// --------------------------------------------------------------------------------------------
// Token-tiled GEMM ([P1] Q1_MM4_WGSL: each weight word decoded once for T tokens, past the last
// token the column is clamped, computed and never stored).  One thread block = one 128-row tile
// (4 warps x 32 rows, one row per lane) x kTok tokens; all blocks of the tile stream through a
// shared ring; the activation constants (DP4A) or tables (LUT4) of the block's sub-blocks are
// built per block by the thread block itself.
// --------------------------------------------------------------------------------------------
constexpr int kTok = 4;
constexpr int kFewTokens = 8;              // DP4A GEMMs up to this many tokens run as per-column GEMVs
constexpr int kGemmStages = 4;

// LUT4: table[t][k][l][nib] = d1 * s(nib) for the 4 activations of lane l, with the nibble's bit
// c (c = 0..3) the sign bit of weight 4l+c.  p = d1 * s is exact.
__device__ __forceinline__ void lut_table(const uint16_t* blk, int l, float* table16) {
    const float d1 = f16_to_f32(blk[0]);
    const uint32_t qw = static_cast<uint32_t>(blk[1 + 2 * l]) | (static_cast<uint32_t>(blk[2 + 2 * l]) << 16);
    int pos[4], neg[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int q = static_cast<int>(static_cast<int8_t>((qw >> (8 * c)) & 0xFFu));
        pos[c] = q;
        neg[c] = (q == -128) ? -128 : -q;
    }
#pragma unroll
    for (int nib = 0; nib < 16; ++nib) {
        int s = 0;
#pragma unroll
        for (int c = 0; c < 4; ++c) s += ((nib >> c) & 1) ? pos[c] : neg[c];
        table16[nib] = __fmul_rn(d1, static_cast<float>(s));
    }
}

// nibble of lane l from a transposed sign word: bits l, 8+l, 16+l, 24+l -> bits 0..3
__device__ __forceinline__ uint32_t lane_nibble(uint32_t w, int l) {
    return (((w >> l) & 0x01010101u) * 0x01020408u) >> 24;
}

template <int kPath>
__global__ void __launch_bounds__(128)
q1_gemm_kernel(const uint8_t* __restrict__ packed, const uint8_t* __restrict__ act, float* __restrict__ y,
               int rows, int n, int cols) {
    __shared__ __align__(128) uint8_t ring[kGemmStages][kChunkBytes];
    __shared__ uint64_t bars[kGemmStages];
    // per token and sub-block: DP4A constants (24 words) or LUT4 tables (8 x 16 floats)
    // LUT4: eight tables of 16 entries, 17 words apart, so that the 32 builders of a token (one
    // (sub-block, lane) table each) store to distinct banks; a lookup reads 16 words of one table
    constexpr int kLutStride = 17;
    constexpr int kPerTokK = (kPath == GQ_PATH_LUT4) ? 8 * kLutStride : kConstWords;
    __shared__ __align__(16) uint32_t tabs[2][kTok][4][kPerTokK];

    const int nb = n / 128;
    const int tile = blockIdx.x;
    const int c0 = blockIdx.y * kTok;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rr = warp * 32 + lane;      // row within the tile
    const uint8_t* tile_base = packed + static_cast<size_t>(tile) * nb * kChunkBytes;
    const size_t act_bytes = static_cast<size_t>(n / 32) * 34;

    if (tid == 0) {
        for (int s = 0; s < kGemmStages; ++s) mbar_init(&bars[s], 1);
        fence_barrier_init();
        const int first = nb < kGemmStages ? nb : kGemmStages;
        for (int s = 0; s < first; ++s) {
            mbar_arrive_expect_tx(&bars[s], kChunkBytes);
            bulk_g2s(ring[s], tile_base + static_cast<size_t>(s) * kChunkBytes, kChunkBytes, &bars[s]);
        }
    }

    float2 acc[kTok][4];
#pragma unroll
    for (int t = 0; t < kTok; ++t)
#pragma unroll
        for (int p = 0; p < 4; ++p) acc[t][p] = make_float2(0.0f, 0.0f);

    for (int i = 0; i < nb; ++i) {
        const int buf = i & 1;
        // build this block's per-token data: kTok tokens x 4 sub-blocks x 8 lanes = 128 items
        {
            const int t = tid >> 5, k = (tid >> 3) & 3, l = tid & 7;
            const int c = min(c0 + t, cols - 1);
            const uint16_t* blk = reinterpret_cast<const uint16_t*>(act + c * act_bytes + static_cast<size_t>(4 * i + k) * 34);
            if (kPath == GQ_PATH_LUT4) {
                lut_table(blk, l, reinterpret_cast<float*>(&tabs[buf][t][k][l * kLutStride]));
            } else {
                uint32_t qt, seed;
                float d1s;
                act_lane_consts(blk, l, qt, seed, d1s);
                tabs[buf][t][k][l] = qt;
                tabs[buf][t][k][8 + l] = seed;
                tabs[buf][t][k][16 + l] = __float_as_uint(d1s);
            }
        }
        __syncthreads();    // tables of block i visible; ring stage of block i-1 fully read
        const int s = i % kGemmStages;
        if (tid == 0 && i >= 1 && i - 1 + kGemmStages < nb) {
            const int sp = (i - 1) % kGemmStages;
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&bars[sp], kChunkBytes);
            bulk_g2s(ring[sp], tile_base + static_cast<size_t>(i - 1 + kGemmStages) * kChunkBytes, kChunkBytes,
                     &bars[sp]);
        }
        const bool ok = __syncthreads_and(mbar_wait(&bars[s], static_cast<uint32_t>(i / kGemmStages) & 1u));
        if (!ok) {
            if (tid == 0) {
                report_error(kErrWaitTimeout);
                const int last = (i + kGemmStages < nb ? i + kGemmStages : nb);
                for (int b = i; b < last; ++b)
                    if (!mbar_wait(&bars[b % kGemmStages], static_cast<uint32_t>(b / kGemmStages) & 1u))
                        report_error(kErrDrainTimeout);
            }
            __syncthreads();
            return;
        }
        const uint4 wb = reinterpret_cast<const uint4*>(ring[s])[rr];
        const float d0 = f16_to_f32(reinterpret_cast<const uint16_t*>(ring[s] + kTileRows * 16)[rr]);
        const float2 dd = make_float2(d0, d0);

#pragma unroll
        for (int t = 0; t < kTok; ++t) {
            float2 ab[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t w = (k == 0) ? wb.x : (k == 1) ? wb.y : (k == 2) ? wb.z : wb.w;
                if (kPath == GQ_PATH_LUT4) {
                    const float* tb = reinterpret_cast<const float*>(&tabs[buf][t][k][0]);
#pragma unroll
                    for (int p = 0; p < 4; ++p) {
                        const float2 v = make_float2(tb[(2 * p) * kLutStride + lane_nibble(w, 2 * p)],
                                                     tb[(2 * p + 1) * kLutStride + lane_nibble(w, 2 * p + 1)]);
                        ab[p] = (k == 0) ? v : fadd2(v, ab[p]);
                    }
                } else {
                    const uint4* cs = reinterpret_cast<const uint4*>(&tabs[buf][t][k][0]);
                    const uint4 q0 = cs[0], q1 = cs[1], s0 = cs[2], s1 = cs[3], e0 = cs[4], e1 = cs[5];
                    float2 tv[4];
                    lane_values(w, q0, q1, s0, s1, tv);
                    const float2 D[4] = {make_float2(__uint_as_float(e0.x), __uint_as_float(e0.y)),
                                         make_float2(__uint_as_float(e0.z), __uint_as_float(e0.w)),
                                         make_float2(__uint_as_float(e1.x), __uint_as_float(e1.y)),
                                         make_float2(__uint_as_float(e1.z), __uint_as_float(e1.w))};
#pragma unroll
                    for (int p = 0; p < 4; ++p) ab[p] = (k == 0) ? fmul2(D[p], tv[p]) : ffma2(D[p], tv[p], ab[p]);
                }
            }
#pragma unroll
            for (int p = 0; p < 4; ++p) acc[t][p] = ffma2(dd, ab[p], acc[t][p]);
        }
    }

    const int row = tile * kTileRows + rr;
#pragma unroll
    for (int t = 0; t < kTok; ++t) {
        const int c = c0 + t;
        if (c < cols && row < rows) y[static_cast<size_t>(c) * rows + row] = final_reduce(acc[t]);
    }
}

}  // namespace

// --------------------------------------------------------------------------------------------
GQ_ERROR_ACCESSOR(q1)

cudaError_t launch_q1_pack(const void* raw, int rows, int n, void* packed, cudaStream_t s) {
    const int nb = n / 128;
    const long long tiles = (rows + kTileRows - 1) / kTileRows;
    const long long total = tiles * nb * kTileRows;
    const int threads = 256;
    const long long blocks = (total + threads - 1) / threads;
    q1_pack_kernel<<<static_cast<unsigned>(blocks), threads, 0, s>>>(static_cast<const uint8_t*>(raw), rows, nb,
                                                                     static_cast<uint8_t*>(packed), total);
    return cudaGetLastError();
}

int gemv_tiles_for(int rows) { return (rows + kTileRows - 1) / kTileRows; }

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

cudaError_t launch_q1_gemv(const void* packed, const void* act, float* y, int rows, int n, void* workspace,
                           int act_format, cudaStream_t s) {
    const int tiles = gemv_tiles_for(rows);
    static int sm_cached[64] = {0};
    int dev = 0;
    cudaError_t e0 = cudaGetDevice(&dev);
    if (e0 != cudaSuccess) return e0;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (sm_cached[dev] == 0) {
        e0 = cudaDeviceGetAttribute(&sm_cached[dev], cudaDevAttrMultiProcessorCount, dev);
        if (e0 != cudaSuccess) return e0;
    }
    if (tiles < sm_cached[dev]) {
        // fewer tiles than SMs: the block-parallel kernel (one launch, no workspace)
        const dim3 grid((rows + 31) / 32), block(kSmallWarps * 32);
        const uint8_t* pw = static_cast<const uint8_t*>(packed);
        const uint8_t* pa = static_cast<const uint8_t*>(act);
        const int nb = n / 128;
        if (act_format == GQ_ACT_F32)
            return nb <= kSmallPass
                       ? launch_dependent(q1_gemv_small_kernel<GQ_ACT_F32, 2>, grid, block, s, pw, pa, y, rows, nb)
                       : launch_dependent(q1_gemv_small_kernel<GQ_ACT_F32, 4>, grid, block, s, pw, pa, y, rows, nb);
        return nb <= kSmallPass
                   ? launch_dependent(q1_gemv_small_kernel<GQ_ACT_Q8_0, 2>, grid, block, s, pw, pa, y, rows, nb)
                   : launch_dependent(q1_gemv_small_kernel<GQ_ACT_Q8_0, 4>, grid, block, s, pw, pa, y, rows, nb);
    }
    int grid = 0, active = 0;
    cudaError_t e = gemv_grid(tiles, &grid, &active);
    if (e != cudaSuccess) return e;
    int* counter = reinterpret_cast<int*>(static_cast<uint8_t*>(workspace) + gemv_workspace_bytes(n) - 16);
    gq_gemv_desc d{packed, act, y, workspace, rows, n, 0, act_format};
    act_prep_kernel<<<dim3(8, 1), 256, 0, s>>>(d, nullptr, 0, counter);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_gemv_dependent(grid, s, GemvArgs{d, nullptr, 0, tiles, active, counter});
}

cudaError_t launch_q1_gemv_grouped(const gq_gemv_desc* descs, int count, int total_tiles, int* counter,
                                   cudaStream_t s) {
    int grid = 0, active = 0;
    cudaError_t e = gemv_grid(total_tiles, &grid, &active);
    if (e != cudaSuccess) return e;
    gq_gemv_desc none{nullptr, nullptr, nullptr, nullptr, 0, 128, 0, 0};
    act_prep_kernel<<<dim3(8, count), 256, 0, s>>>(none, descs, count, counter);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_gemv_dependent(grid, s, GemvArgs{none, descs, count, total_tiles, active, counter});
}

cudaError_t launch_q1_gemm(const void* packed, const void* act, float* y, int rows, int n, int cols, int path,
                           cudaStream_t s) {
    if (path == GQ_PATH_DP4A && cols <= kFewTokens) {
        // a few tokens: each column is a GEMV in the same order, and the single-matrix GEMV kernel
        // spreads 32-row tiles over the GPU (the 4-token tiles below would leave most SMs idle)
        const dim3 grid((rows + 31) / 32, cols), block(kSmallWarps * 32);
        const uint8_t* pw = static_cast<const uint8_t*>(packed);
        const uint8_t* pa = static_cast<const uint8_t*>(act);
        const int nb = n / 128;
        return nb <= kSmallPass
                   ? launch_dependent(q1_gemv_small_kernel<GQ_ACT_Q8_0, 2>, grid, block, s, pw, pa, y, rows, nb)
                   : launch_dependent(q1_gemv_small_kernel<GQ_ACT_Q8_0, 4>, grid, block, s, pw, pa, y, rows, nb);
    }
    const dim3 grid((rows + kTileRows - 1) / kTileRows, (cols + kTok - 1) / kTok);
    if (path == GQ_PATH_LUT4)
        q1_gemm_kernel<GQ_PATH_LUT4><<<grid, 128, 0, s>>>(static_cast<const uint8_t*>(packed),
                                                          static_cast<const uint8_t*>(act), y, rows, n, cols);
    else
        q1_gemm_kernel<GQ_PATH_DP4A><<<grid, 128, 0, s>>>(static_cast<const uint8_t*>(packed),
                                                          static_cast<const uint8_t*>(act), y, rows, n, cols);
    return cudaGetLastError();
}

}  // namespace gq
