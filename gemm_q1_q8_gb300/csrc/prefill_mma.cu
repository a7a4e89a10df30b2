// Prefill GEMM on the 5th-generation tensor cores (tcgen05, kind::f16 with bf16 operands),
// Bonsai-format 1-bit weights x Q8_0 activations, bit-identical to the fixed order
//   S = sum_t (bit ? q : -q) per 32-block, p = f16(xd[m,b]) * S (exact), acc = fma(w_scale[n,b], p, acc).
// (BonsaiのWebGPUカーネルを読み解く: the prefill figure names a cooperative-matrix path beside
// LUT4; this is its sm_103a counterpart.)
//
// The tensor cores compute p itself.  The activation operand is pv = f16(d)*q split exactly into
// three bf16 parts (hi + mid + lo = pv, written by the quantizer, one plane each); the weights are
// +-1, exact in bf16.  Every product is exact, and every term and partial sum of a 32-block's
// p = sum_t (+-1) * (hi + mid + lo) is an integer multiple of the ulp of f16(d) and below 2^12
// times f16(d) in magnitude, so it has at most 23 significant bits and the f32 accumulation is
// exact: the result is
// p = f16(d) * S whatever the order of the additions.  Each 32-block gets its own accumulator
// (3 planes x 2 K=16 MMAs into a fresh TMEM buffer), and the epilogue applies acc = fma(w_s, p, acc)
// in block order: one FP32 operation per block sum (the multiply by dx is gone from it).
//
// Thread block (one per SM): 128 weight rows x 128 tokens, K in stages of 64 (two 32-blocks).
// The weight operand (A, +-1 bf16) lives in tensor memory, written there by the producers with
// tcgen05.st; shared memory holds the activation tiles (B, three planes) and the row-scale ring.
//   warps 0, 1  : MMA issuers (one elected thread each), stages alternating between them, so one
//                 waits on its barriers while the other issues; warp 0 also allocates TMEM
//   warps 2-5   : weight producers, one row per thread (the TMEM lane its warp may write): the
//                 row's two sign words of the stage become 32 columns of +-1 bf16 pairs (u, u+16)
//                 of each 32-block, the order of the quantizer's operand; each thread also writes
//                 its row's two scales of the stage into an 8-slot ring; the first lane starts the
//                 TMA copies of the stage's three activation planes (128-byte swizzle) onto the
//                 same barrier
//   warps 6-21  : epilogue -- per 32-block, two 16x256b tcgen05.ld of the f32 block products p
//                 (each warp its 32 TMEM lanes x 32 columns; a thread holds 4 rows x 8 columns),
//                 acc = fma(w_s, p, acc) in registers; four epilogue warps per SMSP overlap their
//                 TMEM load latencies
// Four stage slots (B 3 x 16 KB of shared memory, A 32 TMEM columns each) and three TMEM
// accumulators of 128 columns, one per 32-block (block b uses accumulator b % 3): each
// accumulator has its own "products ready" and "drained" barriers, so the MMAs of block b + 3
// start as soon as the epilogue has drained block b.  Slot k % 8 of the row-scale ring is written
// again for stage k + 8 only after the MMAs of stage k + 4 completed, which needs every epilogue
// warp past block 2k + 6 (block 2k + 9 reuses the accumulator of block 2k + 6): the slot's
// barrier cannot run a phase ahead of an epilogue warp that still has to wait on it.  Every wait
// is bounded (~1 s); a role that gives up raises an abort flag the others honour, and the block
// drains its copies and MMAs and frees TMEM before it exits.
#include "gq_internal.cuh"
#include "tc_common.cuh"
#include "w1a32_mma.cuh"

#include <cuda_bf16.h>

namespace gq {
GQ_ERROR_ACCESSOR(prefill_mma)

namespace {

constexpr int BM = 128;          // weight rows per tile (MMA M, TMEM lanes)
constexpr int BN = 128;          // tokens per tile (MMA N)
constexpr int BK = 64;           // K per stage (two 32-blocks)
constexpr int kStagesM = 4;
constexpr int kAccs = 3;         // TMEM: three 128-column accumulators, one per 32-block in flight
constexpr int kTmemCols = 512;
constexpr int kAColsPerStage = BK / 2;                  // A slot: 64 bf16 per row = 32 columns of pairs
constexpr int kACol0 = kAccs * BN;                      // A slots after the accumulators (384 + 4 x 32)
static_assert(kACol0 + kStagesM * kAColsPerStage <= kTmemCols, "TMEM columns");
constexpr int kPlanes = 3;             // bf16 parts of the activation operand
constexpr int kTileB = BN * BK * 2;    // 16 KB per plane

constexpr int kWarpA0 = 2, kNumAWarps = 4, kWarpE0 = 6, kNumEWarps = 16;
constexpr int kThreads = (kWarpE0 + kNumEWarps) * 32;   // 704
constexpr int kWSlots = 2 * kStagesM;                   // row-scale ring slots
constexpr int kECols = BN / (kNumEWarps / 4);           // 32 token columns per epilogue warp

// instruction descriptor: D f32, A/B bf16, both K-major, N = 128, M = 128 (A from TMEM)
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (0u << 15) | (0u << 16) |
                            (static_cast<uint32_t>(BN >> 3) << 17) | (static_cast<uint32_t>(BM >> 4) << 24);

struct Bars {
    uint64_t full[kStagesM];          // 4 producer-warp arrivals + the copy's expect_tx arrival, and its bytes
    uint64_t done[kStagesM];          // a stage's MMAs complete: its slots are free
    uint64_t bdone[kAccs];            // a block's MMAs complete: its sums are in its accumulator
    uint64_t tempty[kAccs];           // an accumulator drained by the epilogue
    uint64_t wfull[2 * kStagesM];     // a row-scale slot written by the producers
    uint64_t final_;                  // both issuers' last MMAs have completed
    int last_copy_stage[kStagesM];    // the last stage whose activation copy went into each slot
    uint32_t tmem_base;
    int abort;
};



__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(kIdesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 16 lanes x 32 columns of f32 from TMEM (16x256b shape, four 8-column repetitions): thread t gets,
// per repetition r, rows (t / 4) and (t / 4) + 8 of the 16 at columns 8 r + 2 (t % 4) and + 1, as
// v[4 r .. 4 r + 3] = (row, c), (row, c + 1), (row + 8, c), (row + 8, c + 1).
__device__ __forceinline__ void tc_ld16x256_x4(uint32_t taddr, float* v) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x4.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}



__global__ void __launch_bounds__(kThreads, 1)   // 22 warps: at most 80 registers (6 warps on an SMSP)
prefill_mma_kernel(const __grid_constant__ CUtensorMap tmB, const uint32_t* __restrict__ signs,
                   const float* __restrict__ ws, float* __restrict__ y, int M, int N,
                   int K) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* base = smem_align1024(smem_raw);
    uint8_t* sB = base;                                   // [kStagesM][kPlanes][kTileB]
    Bars* bars = reinterpret_cast<Bars*>(sB + kStagesM * kPlanes * kTileB);
    float* sws = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bars) + ((sizeof(Bars) + 15) & ~size_t(15)));
    volatile int* abort = &bars->abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * BM, m0 = blockIdx.y * BN;
    const int nbk = K / 32;
    const int stages = K / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStagesM; ++s) {
            mbar_init(&bars->full[s], kNumAWarps + 1);
            mbar_init(&bars->done[s], 1);
            bars->last_copy_stage[s] = -1;
        }
        for (int p = 0; p < kAccs; ++p) {
            mbar_init(&bars->bdone[p], 1);
            mbar_init(&bars->tempty[p], kNumEWarps);
        }
        for (int w = 0; w < kWSlots; ++w) mbar_init(&bars->wfull[w], kNumAWarps);
        mbar_init(&bars->final_, 2);
        bars->abort = 0;
        fence_barrier_init();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&bars->tmem_base)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp < kWarpA0) {
        // ---------------- MMA issuers: issuer j takes stages j, j + 2, ...; a commit per block,
        // then one per stage
        if (lane == 0) {
            bool live = true;
            for (int k = warp; k < stages && live && !*abort; k += 2) {
                const int s = k % kStagesM;
                if (!wait_or_abort(&bars->full[s], static_cast<uint32_t>(k / kStagesM) & 1u, abort)) break;
                const uint32_t aslot = tmem + static_cast<uint32_t>(kACol0 + s * kAColsPerStage);
#pragma unroll
                for (int bi = 0; bi < 2; ++bi) {
                    const int b = 2 * k + bi;
                    const int acc = b % kAccs;
                    if (b >= kAccs &&
                        !wait_or_abort(&bars->tempty[acc], static_cast<uint32_t>(b / kAccs - 1) & 1u, abort)) {
                        live = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem + static_cast<uint32_t>(acc * BN);
#pragma unroll
                    for (int p = 0; p < kPlanes; ++p)
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            const int koff = (bi * 32 + j * 16) * 2;     // bytes along the 128-byte row
                            tc_mma_ts(d, aslot + static_cast<uint32_t>(bi * 16 + j * 8),
                                      smem_desc(sB + (s * kPlanes + p) * kTileB + koff), (p | j) ? 1u : 0u);
                        }
                    tc_commit(&bars->bdone[acc]);
                }
                if (live) tc_commit(&bars->done[s]);
            }
            // all MMAs issued so far complete before TMEM may be freed
            tc_commit(&bars->final_);
        }
    } else if (warp < kWarpE0) {
        // ---------------- weight producers: +-1 bf16 pairs into the stage's TMEM slot, one row per
        // thread.  The row's two sign words and two scales per stage are loaded two stages ahead,
        // 8 bytes each (rows are 8-byte aligned: K is a multiple of 64, the arrays 16-byte aligned).
        const int r = (warp & 3) * 32 + lane;                       // row = the TMEM lane this warp may write
        const bool copier = warp == kWarpA0 && lane == 0;
        const int n = min(n0 + r, N - 1);
        const uint2* srow2 = reinterpret_cast<const uint2*>(signs + static_cast<size_t>(n) * nbk);
        const float2* wrow2 = reinterpret_cast<const float2*>(ws + static_cast<size_t>(n) * nbk);
        const uint32_t tlane = static_cast<uint32_t>((warp & 3) * 32) << 16;
        if (copier) prefetch_tmap(&tmB);
        constexpr int kAhead = 2;
        uint2 pf[kAhead];
        float2 pw[kAhead];
#pragma unroll
        for (int a = 0; a < kAhead; ++a) {
            pf[a] = (a < stages) ? __ldg(srow2 + a) : make_uint2(0u, 0u);
            pw[a] = (a < stages) ? __ldg(wrow2 + a) : make_float2(0.0f, 0.0f);
        }
        bool live = true;
        for (int k0 = 0; k0 < stages && live; k0 += kAhead) {
#pragma unroll
            for (int kk = 0; kk < kAhead; ++kk) {
                const int k = k0 + kk;
                if (k >= stages) break;
                const int s = k % kStagesM;
                if (k >= kStagesM &&
                    !wait_or_abort(&bars->done[s], static_cast<uint32_t>(k / kStagesM - 1) & 1u, abort)) {
                    live = false;
                    break;
                }
                if (copier) {
                    mbar_arrive_expect_tx(&bars->full[s], kPlanes * kTileB);
                    for (int p = 0; p < kPlanes; ++p)
                        tma_load_2d(sB + (s * kPlanes + p) * kTileB, &tmB, k * BK, p * M + m0, &bars->full[s]);
                    bars->last_copy_stage[s] = k;
                }
                const uint32_t w2[2] = {pf[kk].x, pf[kk].y};
                pf[kk] = (k + kAhead < stages) ? __ldg(srow2 + k + kAhead) : make_uint2(0u, 0u);
                float* wslot = sws + (k % kWSlots) * 2 * BM;
                wslot[r] = pw[kk].x;
                wslot[BM + r] = pw[kk].y;
                pw[kk] = (k + kAhead < stages) ? __ldg(wrow2 + k + kAhead) : make_float2(0.0f, 0.0f);
                uint32_t av[32];
#pragma unroll
                for (int bi = 0; bi < 2; ++bi)
#pragma unroll
                    for (int u = 0; u < 16; ++u)        // pair (u, u+16): bits u and u+16 -> signs of two bf16
                        av[bi * 16 + u] = ((w2[bi] << (15 - u)) & 0x80008000u) ^ 0xBF80BF80u;   // +-1 bf16
                tc_st32(tmem + tlane + static_cast<uint32_t>(kACol0 + s * kAColsPerStage), av);
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&bars->full[s]);
                    mbar_arrive(&bars->wfull[k % kWSlots]);
                }
            }
        }
    } else {
        // ---------------- epilogue: the scale table (overlapping the pipeline's start), then per
        // stage the two block sums of its TMEM pair
        const int q = warp & 3;                        // TMEM lane quadrant of this warp
        const int h = (warp - kWarpE0) >> 2;           // column quarter
        // 16x256b TMEM loads: per 16-lane half and 8-column repetition, thread t holds rows
        // (t / 4) and (t / 4) + 8 of the half at columns 2 (t % 4) and 2 (t % 4) + 1.  So a
        // thread's block sums cover 4 rows x 8 columns, it needs only 8 token scales per block
        // (four 8-byte loads shared by the 8 threads of equal t % 4), and 4 row scales.
        const int rsub = lane >> 2, csub = 2 * (lane & 3);
        int rloc[4];                                   // the thread's rows in the tile
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) rloc[kk] = q * 32 + 16 * (kk >> 1) + 8 * (kk & 1) + rsub;
        float2 acc[4][4];                              // [row][repetition]: columns 8 r + csub, + 1
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) acc[kk][rr] = make_float2(0.0f, 0.0f);
        bool ok = true;
        for (int k = 0; k < stages && ok; ++k) {
            // wfull: the stage's row scales are in the ring
            if (!wait_or_abort(&bars->wfull[k % kWSlots], static_cast<uint32_t>(k / kWSlots) & 1u, abort)) {
                ok = false;
                break;
            }
            const float* wslot = sws + (k % kWSlots) * 2 * BM;
#pragma unroll
            for (int bi = 0; bi < 2; ++bi) {
                const int b = 2 * k + bi;
                const int accx = b % kAccs;
                float wsr[4];
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) wsr[kk] = wslot[bi * BM + rloc[kk]];
                // bdone: the block's sums are in its accumulator
                if (!wait_or_abort_sleep(&bars->bdone[accx], static_cast<uint32_t>(b / kAccs) & 1u, abort)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32 + 16 * hf) << 16) +
                                           static_cast<uint32_t>(accx * BN + h * kECols);
                    float S[16];
                    tc_ld16x256_x4(taddr, S);
                    tc_wait_ld();
#pragma unroll
                    for (int rr = 0; rr < 4; ++rr) {
                        // p = dx * S (exact), then acc = fma(w_s, p, acc): two separate IEEE steps per column
                        const int ka = 2 * hf, kb = 2 * hf + 1;
                        // p = dx * S from the tensor cores, then acc = fma(w_s, p, acc)
                        const float2 pa = make_float2(S[4 * rr], S[4 * rr + 1]);
                        const float2 pb = make_float2(S[4 * rr + 2], S[4 * rr + 3]);
                        acc[ka][rr] = ffma2(make_float2(wsr[ka], wsr[ka]), pa, acc[ka][rr]);
                        acc[kb][rr] = ffma2(make_float2(wsr[kb], wsr[kb]), pb, acc[kb][rr]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->tempty[accx]);
            }
        }
        if (ok) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const int n = n0 + rloc[kk];
                if (n >= N) continue;
#pragma unroll
                for (int rr = 0; rr < 4; ++rr) {
                    const int m = m0 + h * kECols + 8 * rr + csub;
                    if (m < M) y[static_cast<size_t>(m) * N + n] = acc[kk][rr].x;
                    if (m + 1 < M) y[static_cast<size_t>(m + 1) * N + n] = acc[kk][rr].y;
                }
            }
        }
    }

    // ---------------- teardown: outstanding MMAs finish, copies land, TMEM is freed
    __syncwarp();
    if (warp == 0) {
        if (lane == 0 && !mbar_wait(&bars->final_, 0)) report_error(kErrMmaTimeout);
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x == 32 && *abort) {
        // an aborted block may hold activation copies no MMA waited for: the last copy into each
        // slot lands before the block's shared memory goes away
        for (int s = 0; s < kStagesM; ++s) {
            const int k = bars->last_copy_stage[s];
            if (k >= 0 && !mbar_wait(&bars->full[s], static_cast<uint32_t>(k / kStagesM) & 1u))
                report_error(kErrDrainTimeout);
        }
    }
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    __syncthreads();
}

}  // namespace

cudaError_t launch_prefill_mma(const uint32_t* signs, const float* ws, const uint16_t* xd, const uint16_t* xq_op,
                               float* y, int M, int N, int K, cudaStream_t s) {
    (void)xd;                                   // folded into the operand by the quantizer
    CUtensorMap tmB;
    if (!make_tmap_2d(&tmB, xq_op, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, static_cast<uint64_t>(K),
                      static_cast<uint64_t>(kPlanes) * M, static_cast<uint64_t>(K) * 2, BK, BN, true))
        return cudaErrorInvalidValue;
    const size_t smem = 1024 + static_cast<size_t>(kStagesM) * kPlanes * kTileB + ((sizeof(Bars) + 15) & ~size_t(15)) +
                        static_cast<size_t>(kWSlots) * 2 * BM * sizeof(float);
    if (smem > 227 * 1024) return cudaErrorNotSupported;
    static size_t configured = 0;
    if (smem > configured) {
        cudaError_t e = cudaFuncSetAttribute(prefill_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        configured = smem;
    }
    const dim3 grid((N + BM - 1) / BM, (M + BN - 1) / BN);
    prefill_mma_kernel<<<grid, kThreads, smem, s>>>(tmB, signs, ws, y, M, N, K);
    return cudaGetLastError();
}

// x [M, K] f32 -> planes [3][M][K] bf16 in the prefill operand's order: within each 32-block,
// position 2u <- element u, 2u+1 <- element u+16.  hi = bf16(x), mid = bf16(x - hi),
// lo = bf16(x - hi - mid), each rounded to nearest (hi + mid + lo = x for normal x).  One thread
// per pair (u, u+16): a 32-bit store per plane.
__global__ void split_interleave_kernel(const float* __restrict__ x, uint32_t* __restrict__ planes, size_t pairs) {
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < pairs;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const size_t blk = i >> 4;                  // 32-block (row-major over M and K/32)
        const int u = static_cast<int>(i & 15);
        const float v0 = x[blk * 32 + u], v1 = x[blk * 32 + u + 16];
        uint32_t part[3][2];
        const float vv[2] = {v0, v1};
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const __nv_bfloat16 h = __float2bfloat16_rn(vv[e]);
            const float r1 = __fsub_rn(vv[e], __bfloat162float(h));
            const __nv_bfloat16 md = __float2bfloat16_rn(r1);
            const __nv_bfloat16 lo = __float2bfloat16_rn(__fsub_rn(r1, __bfloat162float(md)));
            part[0][e] = __bfloat16_as_ushort(h);
            part[1][e] = __bfloat16_as_ushort(md);
            part[2][e] = __bfloat16_as_ushort(lo);
        }
#pragma unroll
        for (int p = 0; p < kPlanes; ++p) planes[p * pairs + i] = part[p][0] | (part[p][1] << 16);
    }
}

size_t w1a32_mma_workspace_bytes(int M, int K) { return static_cast<size_t>(kPlanes) * M * K * 2; }

cudaError_t launch_w1a32_mma(const uint32_t* signs, const float* ws, const float* x, float* y, int M, int N, int K,
                             void* workspace, cudaStream_t s) {
    const size_t pairs = static_cast<size_t>(M) * K / 2;
    split_interleave_kernel<<<static_cast<unsigned>(std::min<size_t>((pairs + 255) / 256, 8192)), 256, 0, s>>>(
        x, static_cast<uint32_t*>(workspace), pairs);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_prefill_mma(signs, ws, nullptr, static_cast<const uint16_t*>(workspace), y, M, N, K, s);
}

}  // namespace gq
