// Prefill GEMM on the 5th-generation tensor cores (tcgen05, kind::f16), Bonsai-format 1-bit
// weights x Q8_0 activations, bit-identical to the fixed order
//   S = sum_t (bit ? q : -q) per 32-block, p = f16(xd[m,b]) * S (exact), acc = fma(w_scale[n,b], p, acc).
// (BonsaiのWebGPUカーネルを読み解く: the prefill figure names a cooperative-matrix path beside
// LUT4; this is its sm_103a counterpart.)
//
// Why f16 MMA is exact here: the weights are +-1 and the quants |q| <= 127, both exact in f16;
// every product is an integer below 2^7 and a 32-term block sum is at most 4064 < 2^12, so the
// tensor core's f32 accumulation of one block holds S exactly.  Each 32-block gets its own
// accumulator (two K=16 MMAs into a fresh TMEM buffer), drained and applied in block order.
//
// Thread block (one per SM): 128 weight rows x 128 tokens, K in stages of 64 (two 32-blocks).
//   warp 0      : TMA producer of the activation tiles (f16, interleaved, 128-byte swizzle)
//   warp 1      : TMEM allocator and MMA issuer (one elected thread)
//   warps 2-3   : weight producers -- expand sign bits to +-1 f16 in the same swizzled K-major
//                 layout (pairs (u, u+16) of a 32-block in one 32-bit word, the order the
//                 quantizer's MMA operand uses), two rows per thread
//   warps 4-19  : epilogue -- per 32-block, two 16x256b tcgen05.ld of the f32 block sums (each
//                 warp its 32 TMEM lanes x 32 columns; a thread holds 4 rows x 8 columns, so it
//                 reads 8 token scales, not 32), p = dx*S, acc = fma(w_s, p, acc) in registers;
//                 four epilogue warps per SMSP overlap their TMEM load latencies
// Four smem stages (A 16 KB + B 16 KB each) and four TMEM accumulators of 128 columns, one per
// 32-block (block b uses accumulator b % 4): each accumulator has its own "sums ready" and
// "drained" barriers, so the MMAs of block b + 4 start as soon as the epilogue has drained block
// b, and the epilogue of a block overlaps the MMAs of the next three.  The weight producers also
// bring each stage's row scales (2 x 128 f32) into an 8-slot ring, so the epilogue reads them from
// shared memory.  Slot k % 8 is written again for stage k + 8 only after the MMAs of stage k + 4
// completed, which needs every epilogue warp past stage k + 2 (block 2k + 8 reuses the accumulator
// of block 2k + 4): the slot's barrier cannot run a phase ahead of an epilogue warp that still has
// to wait on it.  Every
// wait is bounded (~1 s); a role that gives up raises an abort flag the others honour, and the
// block drains its copies and MMAs and frees TMEM before it exits.
#include "gq_internal.cuh"

namespace gq {
GQ_ERROR_ACCESSOR(prefill_mma)

namespace {

constexpr int BM = 128;          // weight rows per tile (MMA M, TMEM lanes)
constexpr int BN = 128;          // tokens per tile (MMA N)
constexpr int BK = 64;           // K per stage (two 32-blocks)
constexpr int kStagesM = 4;
constexpr int kAccs = 4;         // TMEM: four 128-column accumulators, one per 32-block in flight
constexpr int kTmemCols = 512;
constexpr int kTileA = BM * BK * 2;    // 16 KB
constexpr int kTileB = BN * BK * 2;    // 16 KB

constexpr int kWarpTma = 0, kWarpMma = 1, kWarpA0 = 2, kNumAWarps = 2, kWarpE0 = 4, kNumEWarps = 16;
constexpr int kThreads = (kWarpE0 + kNumEWarps) * 32;   // 640
constexpr int kARowsPerThread = BM / (kNumAWarps * 32);  // 2
constexpr int kWSlots = 2 * kStagesM;                   // row-scale ring slots
constexpr int kECols = BN / (kNumEWarps / 4);           // 32 token columns per epilogue warp

// instruction descriptor: D f32, A/B f16, both K-major, N = 128, M = 128
constexpr uint32_t kIdesc = (1u << 4) | (0u << 7) | (0u << 10) | (0u << 15) | (0u << 16) |
                            (static_cast<uint32_t>(BN >> 3) << 17) | (static_cast<uint32_t>(BM >> 4) << 24);

struct Bars {
    uint64_t fullA[kStagesM], fullB[kStagesM];
    uint64_t done[kStagesM];          // a stage's MMAs complete: its smem stage is free
    uint64_t bdone[kAccs];            // a block's MMAs complete: its sums are in its accumulator
    uint64_t tempty[kAccs];           // an accumulator drained by the epilogue
    uint64_t wfull[2 * kStagesM];     // a row-scale slot written by the producers
    uint64_t final_;
    uint32_t tmem_base;
    int abort;
};

// 64-bit shared-memory matrix descriptor: 128-byte swizzle, K-major, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t smem_desc(const void* p) {
    const uint64_t addr = smem_u32(p);
    uint64_t d = 0;
    d |= (addr >> 4) & 0x3FFFull;               // start address
    d |= static_cast<uint64_t>(1) << 16;        // leading byte offset (unused for swizzled K-major)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;  // stride byte offset: next 8-row group
    d |= static_cast<uint64_t>(1) << 46;        // descriptor version (sm_100 family)
    d |= static_cast<uint64_t>(2) << 61;        // layout: 128-byte swizzle
    return d;
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(kIdesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
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

// Bounded wait that also gives up when another role has raised the abort flag.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        for (int i = 0; i < 16; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (globaltimer_ns() - t0 > 1000000000ull) {
            report_error(kErrMmaTimeout);
            *abort = 1;
            return false;
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1)
prefill_mma_kernel(const __grid_constant__ CUtensorMap tmB, const uint32_t* __restrict__ signs,
                   const float* __restrict__ ws, const uint16_t* __restrict__ xd, float* __restrict__ y, int M, int N,
                   int K) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = base;                                   // [kStagesM][kTileA]
    uint8_t* sB = base + kStagesM * kTileA;               // [kStagesM][kTileB]
    Bars* bars = reinterpret_cast<Bars*>(sB + kStagesM * kTileB);
    float* sws = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bars) + ((sizeof(Bars) + 15) & ~size_t(15)));
    float* sdx = sws + kWSlots * 2 * BM;                  // [slot][bi][row] row scales, then the dx table
    volatile int* abort = &bars->abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * BM, m0 = blockIdx.y * BN;
    const int nbk = K / 32;
    const int stages = K / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStagesM; ++s) {
            mbar_init(&bars->fullA[s], kNumAWarps);
            mbar_init(&bars->fullB[s], 1);
            mbar_init(&bars->done[s], 1);
        }
        for (int p = 0; p < kAccs; ++p) {
            mbar_init(&bars->bdone[p], 1);
            mbar_init(&bars->tempty[p], kNumEWarps);
        }
        for (int w = 0; w < kWSlots; ++w) mbar_init(&bars->wfull[w], kNumAWarps);
        mbar_init(&bars->final_, 1);
        bars->abort = 0;
        fence_barrier_init();
    }
    if (warp == kWarpMma) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&bars->tmem_base)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // the epilogue's scale table: sdx[b * BN + j] = f16(xd[m0 + j, b]) for the tile's tokens
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    int tma_issued = 0;
    if (warp == kWarpTma) {
        // ---------------- activation tiles by TMA
        if (lane == 0) {
            prefetch_tmap(&tmB);
            for (int k = 0; k < stages; ++k) {
                const int s = k % kStagesM;
                if (k >= kStagesM &&
                    !wait_or_abort(&bars->done[s], static_cast<uint32_t>(k / kStagesM - 1) & 1u, abort))
                    break;
                mbar_arrive_expect_tx(&bars->fullB[s], kTileB);
                tma_load_2d(sB + s * kTileB, &tmB, k * BK, m0, &bars->fullB[s]);
                ++tma_issued;
            }
        }
    } else if (warp == kWarpMma) {
        // ---------------- MMA issue (one thread): a commit per block, then one per stage
        if (lane == 0) {
            bool live = true;
            for (int k = 0; k < stages && live && !*abort; ++k) {
                const int s = k % kStagesM;
                const uint32_t ph = static_cast<uint32_t>(k / kStagesM) & 1u;
                if (!wait_or_abort(&bars->fullA[s], ph, abort) || !wait_or_abort(&bars->fullB[s], ph, abort)) break;
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
                    for (int j = 0; j < 2; ++j) {
                        const int koff = (bi * 32 + j * 16) * 2;     // bytes along the 128-byte row
                        tc_mma(d, smem_desc(sA + s * kTileA + koff), smem_desc(sB + s * kTileB + koff), j);
                    }
                    tc_commit(&bars->bdone[acc]);
                }
                if (live) tc_commit(&bars->done[s]);
            }
            // all MMAs issued so far complete before TMEM may be freed
            tc_commit(&bars->final_);
        }
    } else if (warp < kWarpE0) {
        // ---------------- weight producers: +-1 f16, swizzled K-major, rows r and r + 64 per
        // thread.  A row's two sign words and two scales per stage are loaded three stages
        // ahead, 8 bytes each (rows are 8-byte aligned: K is a multiple of 64, the arrays 16-byte
        // aligned).
        const int r0 = threadIdx.x - kWarpA0 * 32;                // 0..63
        const uint2* srow2[kARowsPerThread];
        const float2* wrow2[kARowsPerThread];
#pragma unroll
        for (int i = 0; i < kARowsPerThread; ++i) {
            const int n = min(n0 + r0 + i * 64, N - 1);
            srow2[i] = reinterpret_cast<const uint2*>(signs + static_cast<size_t>(n) * nbk);
            wrow2[i] = reinterpret_cast<const float2*>(ws + static_cast<size_t>(n) * nbk);
        }
        constexpr int kAhead = 3;
        uint2 pf[kARowsPerThread][kAhead];
        float2 pw[kARowsPerThread][kAhead];
#pragma unroll
        for (int i = 0; i < kARowsPerThread; ++i)
#pragma unroll
            for (int a = 0; a < kAhead; ++a) {
                pf[i][a] = (a < stages) ? __ldg(srow2[i] + a) : make_uint2(0u, 0u);
                pw[i][a] = (a < stages) ? __ldg(wrow2[i] + a) : make_float2(0.0f, 0.0f);
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
#pragma unroll
                for (int i = 0; i < kARowsPerThread; ++i) {
                    const int r = r0 + i * 64;
                    const uint32_t w2[2] = {pf[i][kk].x, pf[i][kk].y};
                    pf[i][kk] = (k + kAhead < stages) ? __ldg(srow2[i] + k + kAhead) : make_uint2(0u, 0u);
                    float* wslot = sws + (k % kWSlots) * 2 * BM;
                    wslot[r] = pw[i][kk].x;
                    wslot[BM + r] = pw[i][kk].y;
                    pw[i][kk] = (k + kAhead < stages) ? __ldg(wrow2[i] + k + kAhead) : make_float2(0.0f, 0.0f);
                    uint8_t* tileA = sA + s * kTileA + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
                    for (int bi = 0; bi < 2; ++bi) {
                        const uint32_t w = w2[bi];
#pragma unroll
                        for (int c4 = 0; c4 < 4; ++c4) {
                            uint32_t hw[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int u = c4 * 4 + e;    // pair (u, u+16): bits u and u+16 -> signs of two f16
                                hw[e] = ((w << (15 - u)) & 0x80008000u) ^ 0xBC00BC00u;
                            }
                            const int chunk = bi * 4 + c4;
                            *reinterpret_cast<uint4*>(tileA + ((chunk ^ (r & 7)) << 4)) =
                                make_uint4(hw[0], hw[1], hw[2], hw[3]);
                        }
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&bars->fullA[s]);
                    mbar_arrive(&bars->wfull[k % kWSlots]);
                }
            }
        }
    } else {
        // ---------------- epilogue: the scale table (overlapping the pipeline's start), then per
        // stage the two block sums of its TMEM pair
        {
        // Two scales (one 32-bit word) per load, consecutive threads on consecutive tokens so the
        // transposed stores are conflict-free; eight independent loads in flight per thread.
        const int t = threadIdx.x - kWarpE0 * 32;
        const int pairs = nbk / 2;                            // nbk is even (K % 64 == 0)
        const int total = pairs * BN;
        for (int base_i = t; base_i < total; base_i += 8 * kNumEWarps * 32) {
            uint32_t v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int idx = base_i + u * kNumEWarps * 32;
                if (idx < total) {
                    const int j = idx % BN, bp = idx / BN;
                    const int m = min(m0 + j, M - 1);
                    v[u] = __ldg(reinterpret_cast<const uint32_t*>(xd + static_cast<size_t>(m) * nbk) + bp);
                }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int idx = base_i + u * kNumEWarps * 32;
                if (idx < total) {
                    const int j = idx % BN, bp = idx / BN;
                    sdx[(2 * bp) * BN + j] = f16_to_f32(v[u] & 0xFFFFu);
                    sdx[(2 * bp + 1) * BN + j] = f16_to_f32(v[u] >> 16);
                }
            }
        }
        }
        asm volatile("bar.sync 1, %0;" ::"r"(kNumEWarps * 32) : "memory");
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
                float2 dxp[4];
#pragma unroll
                for (int rr = 0; rr < 4; ++rr)
                    dxp[rr] = *reinterpret_cast<const float2*>(sdx + b * BN + h * kECols + 8 * rr + csub);
                // bdone: the block's sums are in its accumulator
                if (!wait_or_abort(&bars->bdone[accx], static_cast<uint32_t>(b / kAccs) & 1u, abort)) {
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
                        const float2 pa = fmul2(dxp[rr], make_float2(S[4 * rr], S[4 * rr + 1]));
                        const float2 pb = fmul2(dxp[rr], make_float2(S[4 * rr + 2], S[4 * rr + 3]));
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
    if (warp == kWarpMma) {
        if (lane == 0 && !mbar_wait(&bars->final_, 0)) report_error(kErrMmaTimeout);
        __syncwarp();
    }
    if (warp == kWarpTma && lane == 0) {
        // every activation tile requested must have landed before shared memory is released
        // (on a normal run they were all consumed; after an abort some may still be in flight)
        const int first = tma_issued > kStagesM ? tma_issued - kStagesM : 0;
        for (int k = first; k < tma_issued; ++k)
            if (!mbar_wait(&bars->fullB[k % kStagesM], static_cast<uint32_t>(k / kStagesM) & 1u))
                report_error(kErrDrainTimeout);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWarpMma)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
}

}  // namespace

cudaError_t launch_prefill_mma(const uint32_t* signs, const float* ws, const uint16_t* xd, const uint16_t* xq_op,
                               float* y, int M, int N, int K, cudaStream_t s) {
    CUtensorMap tmB;
    if (!make_tmap_2d(&tmB, xq_op, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, static_cast<uint64_t>(K), static_cast<uint64_t>(M),
                      static_cast<uint64_t>(K) * 2, BK, BN, true))
        return cudaErrorInvalidValue;
    const int nbk = K / 32;
    const size_t smem = 1024 + static_cast<size_t>(kStagesM) * (kTileA + kTileB) + ((sizeof(Bars) + 15) & ~size_t(15)) +
                        static_cast<size_t>(kWSlots) * 2 * BM * sizeof(float) + static_cast<size_t>(nbk) * BN * sizeof(float);
    if (smem > 227 * 1024) return cudaErrorNotSupported;
    static size_t configured = 0;
    if (smem > configured) {
        cudaError_t e = cudaFuncSetAttribute(prefill_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        configured = smem;
    }
    const dim3 grid((N + BM - 1) / BM, (M + BN - 1) / BN);
    prefill_mma_kernel<<<grid, kThreads, smem, s>>>(tmB, signs, ws, xd, y, M, N, K);
    return cudaGetLastError();
}

}  // namespace gq
