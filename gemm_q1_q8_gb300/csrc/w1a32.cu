// Bonsai decode GEMV over f32 activations on sm_103a (BonsaiのWebGPUカーネルを読み解く, the
// decode/prefill figure: llama-decode-q1-proj.wgsl).  The weights are the Bonsai format -- one u32
// of 32 sign bits (bit 1 -> +1.0, bit 0 -> -1.0) and one f32 scale per 32 weights -- and
//   y[m, n] = sum_b ws[n, b] * sum_t s(n, 32 b + t) * x[m, 32 b + t].
// The page leaves the order of the float operations open (it takes dot(x4, s4) per four weights
// and adds scale * d into acc); here each lane sums a block's 32 signed activations in order, then
// acc = fma(scale, d, acc) over its blocks, and a butterfly over the warp's lanes adds the lanes.
//
// As on the page, one activation read serves four rows: a warp covers four weight rows, each lane
// the blocks lane, lane + 32, ... of those rows.  The activations sit in shared memory transposed
// ([t][block], stride odd) so the lanes' reads of consecutive blocks are conflict-free; the sign is
// applied by flipping the float's sign bit (a row's word shifted so bit t lands on bit 31).
#include "gq_internal.cuh"

namespace gq {
namespace {

constexpr int kRowsPerWarp = 4;
constexpr int kWarps = 8;
constexpr int kRowsPerCta = kRowsPerWarp * kWarps;   // 32
constexpr int kPassBlocks = 256;                     // blocks of activations staged per pass (32 KB)

__global__ void __launch_bounds__(kWarps * 32)
q1s32_f32_gemv_kernel(const uint32_t* __restrict__ signs, const float* __restrict__ ws, const float* __restrict__ x,
                      float* __restrict__ y, int N, int K) {
    __shared__ float xs[32 * (kPassBlocks + 1)];     // [t][block], stride kPassBlocks + 1
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m = blockIdx.y;
    const int n0 = blockIdx.x * kRowsPerCta + warp * kRowsPerWarp;
    const int nbk = K / 32;
    const float* xm = x + static_cast<size_t>(m) * K;
    const uint32_t* srow[kRowsPerWarp];
    const float* wrow[kRowsPerWarp];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        const int n = min(n0 + r, N - 1);            // past-the-end rows: computed, not stored
        srow[r] = signs + static_cast<size_t>(n) * nbk;
        wrow[r] = ws + static_cast<size_t>(n) * nbk;
    }
    float acc[kRowsPerWarp];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) acc[r] = 0.0f;

    for (int b0 = 0; b0 < nbk; b0 += kPassBlocks) {
        const int nb = min(kPassBlocks, nbk - b0);
        __syncthreads();
        for (int e = threadIdx.x; e < nb * 32; e += blockDim.x) {   // coalesced reads of x
            const int bl = e >> 5, t = e & 31;
            xs[t * (kPassBlocks + 1) + bl] = xm[static_cast<size_t>(b0) * 32 + e];
        }
        __syncthreads();
        // the rows' words and scales of the lane's next block load while this one is summed
        uint32_t nword[kRowsPerWarp];
        float nsc[kRowsPerWarp];
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
            nword[r] = (lane < nb) ? __ldg(srow[r] + b0 + lane) : 0u;
            nsc[r] = (lane < nb) ? __ldg(wrow[r] + b0 + lane) : 0.0f;
        }
        for (int bl = lane; bl < nb; bl += 32) {
            uint32_t word[kRowsPerWarp];
            float sc[kRowsPerWarp];
#pragma unroll
            for (int r = 0; r < kRowsPerWarp; ++r) {
                word[r] = ~nword[r];                        // inverted: a set bit now marks -1
                sc[r] = nsc[r];
                if (bl + 32 < nb) {
                    nword[r] = __ldg(srow[r] + b0 + bl + 32);
                    nsc[r] = __ldg(wrow[r] + b0 + bl + 32);
                }
            }
            float d[kRowsPerWarp];
#pragma unroll
            for (int r = 0; r < kRowsPerWarp; ++r) d[r] = 0.0f;
#pragma unroll
            for (int t = 0; t < 32; ++t) {
                const uint32_t xv = __float_as_uint(xs[t * (kPassBlocks + 1) + bl]);
#pragma unroll
                for (int r = 0; r < kRowsPerWarp; ++r)
                    d[r] = __fadd_rn(d[r], __uint_as_float(xv ^ ((word[r] << (31 - t)) & 0x80000000u)));
            }
#pragma unroll
            for (int r = 0; r < kRowsPerWarp; ++r) acc[r] = __fmaf_rn(sc[r], d[r], acc[r]);
        }
    }
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        float v = acc[r];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
        acc[r] = v;
    }
    if (lane < kRowsPerWarp) {
        float v = acc[0];
#pragma unroll
        for (int r = 1; r < kRowsPerWarp; ++r)
            if (lane == r) v = acc[r];
        const int n = n0 + lane;
        if (n < N) y[static_cast<size_t>(m) * N + n] = v;
    }
}

}  // namespace

cudaError_t launch_q1s32_f32_gemv(const uint32_t* signs, const float* ws, const float* x, float* y, int N, int K,
                                  int M, cudaStream_t s) {
    const dim3 grid((N + kRowsPerCta - 1) / kRowsPerCta, M);
    q1s32_f32_gemv_kernel<<<grid, kWarps * 32, 0, s>>>(signs, ws, x, y, N, K);
    return cudaGetLastError();
}

}  // namespace gq
