// Ternary bitplane GEMV on sm_103a (BonsaiのWebGPUカーネルを読み解く: w = P - N with P/N
// bitplanes, X the binarized activation bitplane, dot = 2*(popc(P&X) - popc(N&X)) - popc(P) +
// popc(N)).
//
// Evaluated as dot = 2*popc((P & X) | (N & ~X)) - popc(P) - popc(N): the two masked sets are
// disjoint when P & N = 0, and a position with both bits set contributes 2 - 2 = 0 either way,
// so this is the same integer for every input -- one LOP3 and one POPC per word and activation.
//
// One thread per weight row; 128-row x 32-word tiles of P and N arrive by TMA with the 128-byte
// swizzle (conflict-free 16-byte reads per row), together with the matching 32 words of every
// activation row of the batch group, through a 3-stage mbarrier ring.
#include "gq_internal.cuh"

namespace gq {
namespace {

constexpr int kRows = 128;
constexpr int kWords = 32;          // words per tile row (128 bytes)
constexpr int kBG = 16;             // activations per pass
constexpr int kStages = 3;
constexpr int kTileBytes = kRows * kWords * 4;     // 16 KB per plane
constexpr int kXBytes = kBG * kWords * 4;          // 2 KB

struct __align__(1024) TernSmem {
    uint8_t P[kStages][kTileBytes];
    uint8_t N[kStages][kTileBytes];
    uint8_t X[kStages][kXBytes];
    uint64_t bars[kStages];
};

__global__ void __launch_bounds__(kRows)
ternary_kernel(const __grid_constant__ CUtensorMap tmP, const __grid_constant__ CUtensorMap tmN,
               const __grid_constant__ CUtensorMap tmX, int32_t* __restrict__ y, int rows, int k, int batch) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    TernSmem& sm = *reinterpret_cast<TernSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int r = threadIdx.x;
    const int row0 = blockIdx.x * kRows;
    const int b0 = blockIdx.y * kBG;
    const int nb = min(kBG, batch - b0);
    const int chunks = k / (32 * kWords);
    const uint32_t stage_bytes = 2 * kTileBytes + static_cast<uint32_t>(kBG) * kWords * 4;

    if (r == 0) {
        prefetch_tmap(&tmP);
        prefetch_tmap(&tmN);
        prefetch_tmap(&tmX);
        for (int s = 0; s < kStages; ++s) mbar_init(&sm.bars[s], 1);
        fence_barrier_init();
        for (int s = 0; s < kStages && s < chunks; ++s) {
            mbar_arrive_expect_tx(&sm.bars[s], stage_bytes);
            tma_load_2d(sm.P[s], &tmP, s * kWords, row0, &sm.bars[s]);
            tma_load_2d(sm.N[s], &tmN, s * kWords, row0, &sm.bars[s]);
            tma_load_2d(sm.X[s], &tmX, s * kWords, b0, &sm.bars[s]);
        }
    }
    __syncthreads();

    int cnt[kBG];
#pragma unroll
    for (int b = 0; b < kBG; ++b) cnt[b] = 0;
    int pn = 0;

    for (int c = 0; c < chunks; ++c) {
        const int s = c % kStages;
        const bool ok = __syncthreads_and(mbar_wait(&sm.bars[s], static_cast<uint32_t>(c / kStages) & 1u));
        if (!ok) {
            if (r == 0) {
                report_error(kErrWaitTimeout);
                const int last = (c + kStages < chunks ? c + kStages : chunks);
                for (int cc = c; cc < last; ++cc)
                    if (!mbar_wait(&sm.bars[cc % kStages], static_cast<uint32_t>(cc / kStages) & 1u))
                        report_error(kErrDrainTimeout);
            }
            __syncthreads();
            return;
        }
        const uint8_t* Pt = sm.P[s];
        const uint8_t* Nt = sm.N[s];
        const uint32_t* Xt = reinterpret_cast<const uint32_t*>(sm.X[s]);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint4 p4 = *reinterpret_cast<const uint4*>(Pt + swz128(r, j));
            const uint4 n4 = *reinterpret_cast<const uint4*>(Nt + swz128(r, j));
            pn += __popc(p4.x) + __popc(p4.y) + __popc(p4.z) + __popc(p4.w);
            pn += __popc(n4.x) + __popc(n4.y) + __popc(n4.z) + __popc(n4.w);
#pragma unroll
            for (int b = 0; b < kBG; ++b) {
                if (b < nb) {
                    const uint4 x4 = *reinterpret_cast<const uint4*>(Xt + b * kWords + 4 * j);
                    cnt[b] += __popc((p4.x & x4.x) | (n4.x & ~x4.x)) + __popc((p4.y & x4.y) | (n4.y & ~x4.y)) +
                              __popc((p4.z & x4.z) | (n4.z & ~x4.z)) + __popc((p4.w & x4.w) | (n4.w & ~x4.w));
                }
            }
        }
        __syncthreads();   // stage s fully read
        if (r == 0 && c + kStages < chunks) {
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&sm.bars[s], stage_bytes);
            tma_load_2d(sm.P[s], &tmP, (c + kStages) * kWords, row0, &sm.bars[s]);
            tma_load_2d(sm.N[s], &tmN, (c + kStages) * kWords, row0, &sm.bars[s]);
            tma_load_2d(sm.X[s], &tmX, (c + kStages) * kWords, b0, &sm.bars[s]);
        }
    }
    const int row = row0 + r;
    if (row < rows) {
#pragma unroll
        for (int b = 0; b < kBG; ++b)
            if (b < nb) y[static_cast<size_t>(b0 + b) * rows + row] = 2 * cnt[b] - pn;
    }
}

}  // namespace

GQ_ERROR_ACCESSOR(ternary)

cudaError_t launch_ternary(const uint32_t* P, const uint32_t* N, const uint32_t* X, int32_t* y, int rows, int k,
                           int batch, cudaStream_t s) {
    CUtensorMap tmP, tmN, tmX;
    const uint64_t words = static_cast<uint64_t>(k) / 32;
    if (!make_tmap_2d(&tmP, P, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, words, rows, words * 4, kWords, kRows, true) ||
        !make_tmap_2d(&tmN, N, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, words, rows, words * 4, kWords, kRows, true) ||
        !make_tmap_2d(&tmX, X, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, words, batch, words * 4, kWords, kBG, false))
        return cudaErrorInvalidValue;
    const size_t smem = sizeof(TernSmem) + 1024;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(ternary_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const dim3 grid((rows + kRows - 1) / kRows, (batch + kBG - 1) / kBG);
    ternary_kernel<<<grid, kRows, smem, s>>>(tmP, tmN, tmX, y, rows, k, batch);
    return cudaGetLastError();
}

}  // namespace gq
