// Batched prefill with Bonsai-format 1-bit weights (one u32 = 32 sign bits, one f32 scale per
// 32 weights; BonsaiのWebGPUカーネルを読み解く, decode/prefill figure) against Q8_0 activations:
// the activation quantizer and the LUT4 GEMM path.
//
// Order per (m, n), blocks b ascending from +0 (bit for bit):
//   S = sum_t (bit ? q : -q) (int8-wrapping negate), p = f16(xd[m,b]) * S (exact),
//   acc = fma(w_scale[n,b], p, acc).
// LUT4 (binary-lut4-matmul): per token and 4 activations, the 16 possible signed sums are
// tabulated once in shared memory; a 4-bit slice of a sign word then picks its partial sum with
// one lookup, and eight lookups make S exactly (integer), shared by every weight row of the tile.
#include "gq_internal.cuh"

#include <cuda_bf16.h>

namespace gq {
namespace {

// ----------------------------------------------------------------------------- quantizer
// A warp takes kQBlocks consecutive 32-blocks, one value per lane of each, all loaded before any
// is quantized (one memory round trip per warp instead of one per block); per block: amax by
// shuffles, d = amax/127, q = round-half-up(x/d) clamped -- every value's arithmetic as before.
constexpr int kQBlocks = 8;

__global__ void __launch_bounds__(256)
quantize_kernel(const float* __restrict__ x, int m, int k, uint16_t* __restrict__ d, int8_t* __restrict__ q,
                uint16_t* __restrict__ op) {
    const long long gw = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const long long nblocks = static_cast<long long>(m) * (k / 32);
    const long long b0 = gw * kQBlocks;
    if (b0 >= nblocks) return;                                  // whole warps only
    float v[kQBlocks];
#pragma unroll
    for (int i = 0; i < kQBlocks; ++i)
        v[i] = (b0 + i < nblocks) ? x[static_cast<size_t>(b0 + i) * 32 + lane] : 0.0f;
    const size_t plane = static_cast<size_t>(m) * k;
#pragma unroll
    for (int i = 0; i < kQBlocks; ++i) {
        if (b0 + i >= nblocks) break;                           // uniform across the warp
        const size_t base = static_cast<size_t>(b0 + i) * 32;   // row * k + b * 32
        float amax = fabsf(v[i]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float dd = q8_0_scale(amax);
        const int qi = q8_0_quant(v[i], amax, dd);
        q[base + lane] = static_cast<int8_t>(qi);
        if (lane == 0) d[b0 + i] = __half_as_ushort(__float2half_rn(dd));
        if (op) {
            // the MMA operand: pv = f16(d) * q (exact: 11 x 7 significant bits), split exactly into
            // three bf16 parts hi = bf16(pv), mid = bf16(pv - hi), lo = bf16(pv - hi - mid) (each
            // rounded to nearest; the subtractions are exact and pv has at most 18 significant bits,
            // so hi + mid + lo = pv), one plane each, the 32-block's elements interleaved
            const int pos = lane < 16 ? 2 * lane : 2 * (lane - 16) + 1;
            const float pv = __fmul_rn(__half2float(__float2half_rn(dd)), static_cast<float>(qi));
            const __nv_bfloat16 hi = __float2bfloat16_rn(pv);
            const float r1 = __fsub_rn(pv, __bfloat162float(hi));
            const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
            const __nv_bfloat16 lo = __float2bfloat16_rn(__fsub_rn(r1, __bfloat162float(mid)));
            op[base + pos] = __bfloat16_as_ushort(hi);
            op[plane + base + pos] = __bfloat16_as_ushort(mid);
            op[2 * plane + base + pos] = __bfloat16_as_ushort(lo);
        }
    }
}

// ----------------------------------------------------------------------------- LUT4 GEMM
constexpr int kTN = 128;   // weight rows per thread block (one per thread)
constexpr int kTM = 32;    // tokens per thread block

__global__ void __launch_bounds__(kTN)
prefill_lut4_kernel(const uint32_t* __restrict__ signs, const float* __restrict__ ws, const uint16_t* __restrict__ xd,
                    const int8_t* __restrict__ xq, float* __restrict__ y, int M, int N, int K) {
    __shared__ __align__(16) int tab[kTM][8][16];     // [token][group][nibble] partial sums
    __shared__ float dx[kTM];
    const int tid = threadIdx.x;
    const int n = blockIdx.x * kTN + tid;
    const int nc = min(n, N - 1);
    const int m0 = blockIdx.y * kTM;
    const int nbk = K / 32;

    float acc[kTM];
#pragma unroll
    for (int t = 0; t < kTM; ++t) acc[t] = 0.0f;

    for (int b = 0; b < nbk; ++b) {
        __syncthreads();
        // kTM tokens x 8 groups = 256 tables, two per thread
#pragma unroll
        for (int it = 0; it < 2; ++it) {
            const int item = tid + it * kTN;
            const int t = item >> 3, g = item & 7;
            const int mc = min(m0 + t, M - 1);
            const uint32_t qw = *reinterpret_cast<const uint32_t*>(xq + static_cast<size_t>(mc) * K + b * 32 + 4 * g);
            int pos[4], neg[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int qv = static_cast<int>(static_cast<int8_t>((qw >> (8 * c)) & 0xFFu));
                pos[c] = qv;
                neg[c] = (qv == -128) ? -128 : -qv;
            }
            int base = neg[0] + neg[1] + neg[2] + neg[3];
            const int delta[4] = {pos[0] - neg[0], pos[1] - neg[1], pos[2] - neg[2], pos[3] - neg[3]};
            int* tb = tab[t][g];
#pragma unroll
            for (int nib = 0; nib < 16; ++nib) {
                int s = base;
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    if ((nib >> c) & 1) s += delta[c];
                tb[nib] = s;
            }
            if (g == 0) dx[t] = f16_to_f32(xd[static_cast<size_t>(mc) * nbk + b]);
        }
        __syncthreads();
        const uint32_t w = __ldg(signs + static_cast<size_t>(nc) * nbk + b);
        const float wsc = __ldg(ws + static_cast<size_t>(nc) * nbk + b);
        int off[8];
#pragma unroll
        for (int g = 0; g < 8; ++g) off[g] = g * 16 + static_cast<int>((w >> (4 * g)) & 0xFu);
        const int* tflat = &tab[0][0][0];
#pragma unroll
        for (int t = 0; t < kTM; ++t) {
            const int* tt = tflat + t * 128;
            const int S = tt[off[0]] + tt[off[1]] + tt[off[2]] + tt[off[3]] + tt[off[4]] + tt[off[5]] +
                          tt[off[6]] + tt[off[7]];
            const float p = __fmul_rn(dx[t], static_cast<float>(S));
            acc[t] = __fmaf_rn(wsc, p, acc[t]);
        }
    }
    if (n < N) {
#pragma unroll
        for (int t = 0; t < kTM; ++t)
            if (m0 + t < M) y[static_cast<size_t>(m0 + t) * N + n] = acc[t];
    }
}

}  // namespace

cudaError_t launch_quantize(const float* x, int m, int k, uint16_t* d, int8_t* q, uint16_t* op, cudaStream_t s) {
    const long long warps = (static_cast<long long>(m) * (k / 32) + kQBlocks - 1) / kQBlocks;
    const long long blocks = (warps * 32 + 255) / 256;
    quantize_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(x, m, k, d, q, op);
    return cudaGetLastError();
}

cudaError_t launch_prefill_lut4(const uint32_t* signs, const float* ws, const uint16_t* xd, const int8_t* xq,
                                float* y, int M, int N, int K, cudaStream_t s) {
    const dim3 grid((N + kTN - 1) / kTN, (M + kTM - 1) / kTM);
    prefill_lut4_kernel<<<grid, kTN, 0, s>>>(signs, ws, xd, xq, y, M, N, K);
    return cudaGetLastError();
}

}  // namespace gq
