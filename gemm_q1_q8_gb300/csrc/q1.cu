// Q1_0 weights x Q8_0 activations on sm_103a: one-time repack, the single-matrix decode GEMV for
// matrices with fewer tiles than SMs, and the token-tiled GEMM (DP4A and LUT4 paths).  The grouped
// layer sweep and the persistent GEMV are in q1_gemv.cu; the arithmetic they share, in
// q1_common.cuh.
#include "q1_common.cuh"

namespace gq {

namespace {

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
    return launch_q1_gemv_persistent(packed, act, y, rows, n, workspace, act_format, s);
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
