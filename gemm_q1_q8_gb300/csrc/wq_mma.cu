// W8A32 and W4A32 group-128 matmuls on the 5th-generation tensor cores (web-xpu-ops README:
// matmulQ8 -- int8 weights [N, K] with one f32 scale per row; matmulQ4G128 -- 4-bit weights with one
// f32 scale per 128 columns; f32 activations [T, K]):
//   8 bits: y[t, n] = scale[n] * sum_k q[n, k] x[t, k]
//   4 bits: y[t, n] = sum_g scale[n, g] * sum_{k in g} q[n, k] x[t, k]
//
// The activations are f32, the tensor cores take bf16: each x is split exactly into three bf16
// parts, hi = bf16(x), mid = bf16(x - hi), lo = bf16(x - hi - mid) (round to nearest each time; the
// two subtractions are exact), so hi + mid + lo = x for every normal x.  The int8 codes are exact in
// bf16.  Every product code * part is exact in the tensor core.  The three parts of one 128-column
// round (two 64-column smem stages, 24 MMA steps) accumulate into a TMEM accumulator of their own;
// the epilogue adds the round partials in round order in f32 with round to nearest and multiplies
// by the row scale at the end (8 bits), or folds each partial in with one fma by the scale of its
// group (4 bits: a round is exactly one 128-column group).  (The tensor core's own f32 accumulation
// is not round-to-nearest: letting one accumulator run over all of K gave a one-signed error that
// grew with K.)
//
// Thread block (one per SM): 128 weight rows x 128 tokens, K in stages of 64.  The weight operand
// (A) lives in tensor memory, written there by the producers with tcgen05.st; shared memory holds
// only the activation planes (B), so the MMAs' shared-memory reads are B's alone.
//   warps 0, 1  : MMA issuers (one elected thread each), rounds alternating between them, so one
//                 waits on its barriers while the other keeps the tensor pipe fed; warp 0 also
//                 allocates and frees TMEM
//   warps 2-5   : producer group 0 (even stages), warps 6-9: group 1 (odd stages): one weight row
//                 per thread (the TMEM lane its warp may write), the row's 64 codes of the stage
//                 become 32 columns of bf16 pairs in the stage's A slot; each thread fetches its
//                 row's codes two of its stages ahead with cp.async into a private shared-memory
//                 ring (no registers held, no barrier: only the thread reads what it copied); the
//                 group's first lane also starts the TMA copy of the three activation planes of the
//                 stage (128B swizzle) onto the same barrier
//   warps 10-17 : epilogue: after every round, tcgen05.ld of its accumulator (a warp holds 32 rows
//                 x 64 tokens) added into registers; at the end y = scale * sum
// Four stage slots (B 3 x 16 KB in shared memory, A 32 TMEM columns each), three TMEM
// accumulators of 128 columns, 32 KB of code rings.  The kernel is launched as a programmatic
// dependent of the split: everything but the activation copies starts before the split finishes.  Every wait is bounded (~1 s); a role that gives up raises an abort
// flag the others honour, and the block drains its copies and MMAs and frees TMEM before it exits.
#include "gq_internal.cuh"
#include "tc_common.cuh"
#include "wq_mma.cuh"

#include <cuda_bf16.h>

namespace gq {
GQ_ERROR_ACCESSOR(wq_mma)

namespace {

constexpr int BM = 128, BN = 128, BK = 64;
constexpr int kStages = 4;
constexpr int kPlanes = 3;
constexpr int kTileB = BN * BK * 2;               // 16 KB per plane
constexpr int kAccs = 3;                          // TMEM accumulators of BN columns, round r -> r % kAccs
constexpr int kAColsPerStage = BK / 2;            // A slot: 64 bf16 per row = 32 columns of pairs
constexpr int kACol0 = kAccs * BN;                // A slots after the accumulators (384 + 4 x 32 = 512)
constexpr int kRoundStages = 2;                   // 64-column stages per round (128 columns)
constexpr int kWarpP0 = 2, kGroupWarps = 4, kWarpE0 = 10, kNumEWarps = 8;
constexpr int kThreads = (kWarpE0 + kNumEWarps) * 32;    // 576
constexpr int kTmemCols = 512;
constexpr int kRing = 2;                          // code-ring slots per producer thread (its stages ahead)
constexpr int kRingBytes = 2 * kRing * 4 * 128 * 16;   // 2 groups x slots x 4 chunks x 128 rows x 16 B
static_assert(kACol0 + kStages * kAColsPerStage <= kTmemCols, "TMEM columns");

// instruction descriptor: D f32, A/B bf16, both K-major, N = 128, M = 128 (A from TMEM)
constexpr uint32_t kIdescBf16 = (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(BN >> 3) << 17) |
                                (static_cast<uint32_t>(BM >> 4) << 24);

struct Bars {
    uint64_t full[kStages];          // 4 producer-warp arrivals + the copy's expect_tx arrival, and its bytes
    uint64_t done[kStages];          // the stage's MMAs have completed (slot free)
    uint64_t accfull[kAccs], accempty[kAccs];
    uint64_t final_;                 // both issuers' last MMAs have completed
    int last_copy_stage[kStages];    // the last stage whose activation copy went into each slot
    uint32_t tmem_base;
    int abort;
};

__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(kIdescBf16), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int kPending>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(kPending) : "memory");
}
__device__ __forceinline__ void tc_ld16(uint32_t taddr, float* v) {    // 32 lanes x 16 columns
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}


// Four int8 codes (a word) as two words of bf16 pairs (codes 0,1 and 2,3), exactly.
__device__ __forceinline__ uint2 codes_to_bf16x4(uint32_t w) {
    const uint32_t b = w ^ 0x80808080u;
    const float2 bias = make_float2(8388736.0f, 8388736.0f);            // 2^23 + 128
    const float2 lo = fadd2(make_float2(__uint_as_float(__byte_perm(b, 0x4B000000u, 0x7440)),
                                        __uint_as_float(__byte_perm(b, 0x4B000000u, 0x7441))),
                            make_float2(-bias.x, -bias.y));
    const float2 hi = fadd2(make_float2(__uint_as_float(__byte_perm(b, 0x4B000000u, 0x7442)),
                                        __uint_as_float(__byte_perm(b, 0x4B000000u, 0x7443))),
                            make_float2(-bias.x, -bias.y));
    // |code| <= 128 has at most 8 significant bits: the upper half of its f32 is its bf16
    return make_uint2(__byte_perm(__float_as_uint(lo.x), __float_as_uint(lo.y), 0x7632),
                      __byte_perm(__float_as_uint(hi.x), __float_as_uint(hi.y), 0x7632));
}

// Eight 4-bit two's-complement codes (a word, nibble 0 first) as four words of bf16 pairs, exactly.
__device__ __forceinline__ uint4 nibbles_to_bf16x8(uint32_t w) {
    const uint32_t b = w ^ 0x88888888u;                  // code + 8 in every nibble
    const uint32_t ev = b & 0x0F0F0F0Fu;                 // codes 0, 2, 4, 6 as bytes
    const uint32_t od = (b >> 4) & 0x0F0F0F0Fu;          // codes 1, 3, 5, 7
    const float2 bias = make_float2(-8388616.0f, -8388616.0f);       // -(2^23 + 8)
    uint32_t out[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t sel = 0x7440u + static_cast<uint32_t>(j);
        const float2 f = fadd2(make_float2(__uint_as_float(__byte_perm(ev, 0x4B000000u, sel)),
                                           __uint_as_float(__byte_perm(od, 0x4B000000u, sel))),
                               bias);
        out[j] = __byte_perm(__float_as_uint(f.x), __float_as_uint(f.y), 0x7632);
    }
    return make_uint4(out[0], out[1], out[2], out[3]);
}

template <int BITS>
__global__ void __launch_bounds__(kThreads, 1)
wq_mma_kernel(const __grid_constant__ CUtensorMap tmB, const uint32_t* __restrict__ w, const float* __restrict__ scale,
              float* __restrict__ y, int T, int N, int K) {
    constexpr int kLd = BITS == 8 ? 4 : 2;               // uint4 loads per row and stage (64 codes)
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // Aligned as an integer on purpose: with the shared-space pointer (smem_align1024) this kernel's
    // 8-bit instance spills under its 96-register budget and measured ~6% slower.
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sB = base;                                      // [kStages][kPlanes][kTileB]
    uint8_t* sC = sB + kStages * kPlanes * kTileB;           // [group][kRing][4 chunks][128 rows] x 16 B
    Bars* bars = reinterpret_cast<Bars*>(sC + kRingBytes);
    volatile int* abort = &bars->abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * BM, t0 = blockIdx.y * BN;
    const int stages = (K + BK - 1) / BK;     // the activation tile past K is zero-filled by the copy
    const int rounds = (stages + kRoundStages - 1) / kRoundStages;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars->full[s], kGroupWarps + 1);
            mbar_init(&bars->done[s], 1);
            bars->last_copy_stage[s] = -1;
        }
        for (int a = 0; a < kAccs; ++a) {
            mbar_init(&bars->accfull[a], 1);
            mbar_init(&bars->accempty[a], kNumEWarps);
        }
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

    if (warp < kWarpP0) {
        // ---------------- MMA issuers: issuer j takes rounds j, j + 2, ...
        if (lane == 0) {
            for (int r = warp; r < rounds && !*abort; r += 2) {
                const int a = r % kAccs;
                if (r >= kAccs &&
                    !wait_or_abort(&bars->accempty[a], static_cast<uint32_t>(r / kAccs - 1) & 1u, abort))
                    break;
                const uint32_t d = tmem + static_cast<uint32_t>(a * BN);
                bool ok = true;
                for (int k = r * kRoundStages; k < min(stages, (r + 1) * kRoundStages); ++k) {
                    const int s = k % kStages;
                    if (!wait_or_abort(&bars->full[s], static_cast<uint32_t>(k / kStages) & 1u, abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const bool first = k == r * kRoundStages;
                    const uint32_t aslot = tmem + static_cast<uint32_t>(kACol0 + s * kAColsPerStage);
#pragma unroll
                    for (int p = 0; p < kPlanes; ++p)
#pragma unroll
                        for (int j = 0; j < BK / 16; ++j)
                            tc_mma_ts(d, aslot + static_cast<uint32_t>(j * 8),
                                      smem_desc(sB + (s * kPlanes + p) * kTileB + j * 32),
                                      (first && p == 0 && j == 0) ? 0u : 1u);
                    tc_commit(&bars->done[s]);
                }
                if (!ok) break;
                tc_commit(&bars->accfull[a]);
            }
            tc_commit(&bars->final_);
        }
    } else if (warp < kWarpE0) {
        // ---------------- producers: group g takes stages g, g + 2, ...
        const int g = (warp - kWarpP0) / kGroupWarps;
        const bool copier = lane == 0 && warp == kWarpP0 + g * kGroupWarps;
        const int r = (warp & 3) * 32 + lane;                   // row = the TMEM lane this warp may write
        const int n = min(n0 + r, N - 1);                       // past-the-end rows: produced, not stored
        const int chunks = K * BITS / 128;                      // uint4s per row; a K % 64 == 32 tail reads zeros
        const uint4* row = reinterpret_cast<const uint4*>(w) + static_cast<size_t>(n) * chunks;
        if (copier) prefetch_tmap(&tmB);
        uint8_t* ring = sC + (g * kRing * 4 * 128 + r) * 16;      // + (slot * 4 + chunk) * 128 * 16
        auto fetch = [&](int kk, int slot) {                     // this thread's codes of stage kk
#pragma unroll
            for (int i = 0; i < kLd; ++i) {
                const int c = kLd * kk + i;
                if (kk < stages && c < chunks) cp_async16(ring + (slot * 4 + i) * 128 * 16, row + c);
            }
            cp_async_commit();
        };
        fetch(g, 0);
        fetch(g + 2, 1);
        const uint32_t tlane = static_cast<uint32_t>((warp & 3) * 32) << 16;
        bool waited = false;                                     // the split has finished (copier only)
        for (int k = g, m = 0; k < stages; k += 2, ++m) {
            const int s = k % kStages;
            if (k >= kStages && !wait_or_abort(&bars->done[s], static_cast<uint32_t>(k / kStages - 1) & 1u, abort))
                break;
            if (copier) {
                if (!waited) {
                    asm volatile("griddepcontrol.wait;" ::: "memory");   // the activation planes are written
                    waited = true;
                }
                mbar_arrive_expect_tx(&bars->full[s], kPlanes * kTileB);
                for (int p = 0; p < kPlanes; ++p)
                    tma_load_2d(sB + (s * kPlanes + p) * kTileB, &tmB, k * BK, p * T + t0, &bars->full[s]);
                bars->last_copy_stage[s] = k;
            }
            cp_async_wait<kRing - 1>();                           // this stage's codes have landed
            const int slot = m % kRing;
            uint4 cw[kLd];
#pragma unroll
            for (int i = 0; i < kLd; ++i)
                cw[i] = (kLd * k + i < chunks) ? *reinterpret_cast<const uint4*>(ring + (slot * 4 + i) * 128 * 16)
                                               : make_uint4(0u, 0u, 0u, 0u);
            uint32_t av[32];                               // bf16 pairs (codes 2i, 2i + 1) of the row
            if constexpr (BITS == 8) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t ws[4] = {cw[i].x, cw[i].y, cw[i].z, cw[i].w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint2 pr = codes_to_bf16x4(ws[j]);
                        av[8 * i + 2 * j] = pr.x;
                        av[8 * i + 2 * j + 1] = pr.y;
                    }
                }
            } else {
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const uint32_t ws[4] = {cw[i].x, cw[i].y, cw[i].z, cw[i].w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint4 pr = nibbles_to_bf16x8(ws[j]);
                        av[16 * i + 4 * j] = pr.x;
                        av[16 * i + 4 * j + 1] = pr.y;
                        av[16 * i + 4 * j + 2] = pr.z;
                        av[16 * i + 4 * j + 3] = pr.w;
                    }
                }
            }
            tc_st32(tmem + tlane + static_cast<uint32_t>(kACol0 + s * kAColsPerStage), av);
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->full[s]);
            fetch(k + 2 * kRing, slot);                          // the slot's codes are consumed
        }
        cp_async_wait<0>();                                      // no copy lands after the block is gone
    } else {
        // ---------------- epilogue: y = scale * (sum over rounds of the round partials) (8 bits), or
        //                  the fma chain of group scale * round partial (4 bits)
        const int q = warp & 3;                                  // TMEM lanes 32q..32q+31
        const int h = (warp - kWarpE0) / 4;                      // tokens 64h..64h+63 of the tile
        const int rr = q * 32 + lane;
        const int n = n0 + rr;
        float acc[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) acc[i] = 0.0f;
        bool ok = true;
        const int groups = (K + 127) / 128;
        const float* gscale = scale + static_cast<size_t>(min(n, N - 1)) * groups;   // 4 bits
        for (int r = 0; r < rounds; ++r) {
            const int a = r % kAccs;
            const float sg = BITS == 4 ? __ldg(gscale + r) : 0.0f;
            if (!wait_or_abort(&bars->accfull[a], static_cast<uint32_t>(r / kAccs) & 1u, abort) || *abort) {
                ok = false;
                break;
            }
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float v[16];
                tc_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(a * BN + h * 64 + c * 16), v);
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    acc[c * 16 + i] = BITS == 8 ? __fadd_rn(acc[c * 16 + i], v[i]) : __fmaf_rn(sg, v[i], acc[c * 16 + i]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->accempty[a]);
        }
        if (ok && n < N) {
            const float sc = BITS == 8 ? __ldg(scale + n) : 1.0f;
#pragma unroll
            for (int i = 0; i < 64; ++i) {
                const int t = t0 + h * 64 + i;
                if (t < T) y[static_cast<size_t>(t) * N + n] = BITS == 8 ? __fmul_rn(sc, acc[i]) : acc[i];
            }
        }
    }

    // ---------------- teardown
    __syncwarp();
    if (warp == 0) {
        // every MMA issued has completed before TMEM is freed
        if (lane == 0 && !mbar_wait(&bars->final_, 0)) report_error(kErrMmaTimeout);
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x == 32 && *abort) {
        // an aborted block may hold activation copies no MMA waited for: the last copy into each
        // slot lands before the block's shared memory goes away
        for (int s = 0; s < kStages; ++s) {
            const int k = bars->last_copy_stage[s];
            if (k >= 0 && !mbar_wait(&bars->full[s], static_cast<uint32_t>(k / kStages) & 1u))
                report_error(kErrDrainTimeout);
        }
    }
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    __syncthreads();
}

// x [T, K] f32 -> planes [3][T][K] bf16: hi = bf16(x), mid = bf16(x - hi), lo = bf16(x - hi - mid).
__global__ void split_planes_kernel(const float4* __restrict__ x, uint2* __restrict__ planes, size_t quads) {
    // the matmul grid may launch now; its activation copies still wait for this grid's writes
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < quads;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const float4 v = x[i];
        const float vv[4] = {v.x, v.y, v.z, v.w};
        uint32_t h[4], m[4], l[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const __nv_bfloat16 bh = __float2bfloat16_rn(vv[j]);
            const float r1 = __fsub_rn(vv[j], __bfloat162float(bh));
            const __nv_bfloat16 bm = __float2bfloat16_rn(r1);
            const float r2 = __fsub_rn(r1, __bfloat162float(bm));
            const __nv_bfloat16 bl = __float2bfloat16_rn(r2);
            h[j] = __bfloat16_as_ushort(bh);
            m[j] = __bfloat16_as_ushort(bm);
            l[j] = __bfloat16_as_ushort(bl);
        }
        planes[i] = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
        planes[quads + i] = make_uint2(m[0] | (m[1] << 16), m[2] | (m[3] << 16));
        planes[2 * quads + i] = make_uint2(l[0] | (l[1] << 16), l[2] | (l[3] << 16));
    }
}

}  // namespace

size_t wq_mma_workspace_bytes(int T, int K) { return static_cast<size_t>(kPlanes) * T * K * 2; }

cudaError_t launch_wq_mma(int bits, const uint32_t* w, const float* scale, const float* x, float* y, int T, int N,
                          int K, void* workspace, cudaStream_t s) {
    const size_t quads = static_cast<size_t>(T) * K / 4;
    split_planes_kernel<<<static_cast<unsigned>(std::min<size_t>((quads + 255) / 256, 4096)), 256, 0, s>>>(
        reinterpret_cast<const float4*>(x), static_cast<uint2*>(workspace), quads);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    CUtensorMap tmB;
    if (!make_tmap_2d(&tmB, workspace, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, static_cast<uint64_t>(K),
                      static_cast<uint64_t>(kPlanes) * T, static_cast<uint64_t>(K) * 2, BK, BN, true))
        return cudaErrorInvalidValue;
    const size_t smem = 1024 + static_cast<size_t>(kStages) * kPlanes * kTileB + kRingBytes + sizeof(Bars);
    static int configured_dev[2] = {-1, -1};
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    const int b = bits == 8 ? 0 : 1;
    if (configured_dev[b] != dev) {
        e = cudaFuncSetAttribute(bits == 8 ? wq_mma_kernel<8> : wq_mma_kernel<4>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        configured_dev[b] = dev;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((N + BM - 1) / BM, (T + BN - 1) / BN);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = bits == 8 ? cudaLaunchKernelEx(&cfg, wq_mma_kernel<8>, tmB, w, scale, y, T, N, K)
                  : cudaLaunchKernelEx(&cfg, wq_mma_kernel<4>, tmB, w, scale, y, T, N, K);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace gq
