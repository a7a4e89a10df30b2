// block_q8_matmul_nt on sm_103a (kopitiam-gpu block_q8_matmul_nt.wgsl): y = x . w^T with int8
// weights packed four per u32 (little-endian, sign-extended) and one f32 scale per 32-block.
// Order, bit for bit: per (row, col), block b ascending: block_sum = 0; block_sum = block_sum +
// x*q for t = 0..31 (a rounded multiply, then a rounded add); acc = acc + scale*block_sum.
//
// Each thread owns two weight columns and a tile of MT activation rows: the two columns' chains
// run side by side (two scalar round-to-nearest products, then one packed f32x2 add: each lane
// one IEEE operation), the activation tile sits transposed in shared memory (one broadcast load
// feeds four rows), and an int8 becomes an exact f32 as bits 0x4B0000xx (2^23 + q + 128) minus
// 2^23 + 128.  The products stay scalar on purpose: ptxas contracts a packed mul.rn.f32x2 that
// feeds a packed add.rn.f32x2 into one fused fma.rn.f32x2 (observed on sm_103a), which would
// change the rounding of every step; a scalar mul.rn is never contracted.
#include "gq_internal.cuh"

namespace gq {
namespace {

constexpr int kThreads = 256;
constexpr int kKC = 256;                 // activation columns staged per pass (8 blocks)
constexpr float kQBias = 8388736.0f;     // 2^23 + 128

// two rounded products, kept out of any contraction
__device__ __forceinline__ float2 mul_pair(float a, float2 b) {
    return make_float2(__fmul_rn(a, b.x), __fmul_rn(a, b.y));
}

// element j (0..3) of a word already XORed with 0x80808080, as an exact float
__device__ __forceinline__ float q_of(uint32_t u, int j) {
    return __int_as_float(static_cast<int>(__byte_perm(u, 0x4B000000u, 0x7540u | j))) - kQBias;
}

template <int MT>
__global__ void __launch_bounds__(kThreads)
block_q8_kernel(const float* __restrict__ x, const uint32_t* __restrict__ quants, const float* __restrict__ scales,
                float* __restrict__ y, int m, int k, int n) {
    __shared__ __align__(16) float xs[kKC][MT < 4 ? 4 : MT];
    constexpr int MS = MT < 4 ? 4 : MT;
    const int col0 = (blockIdx.x * kThreads + threadIdx.x) * 2;
    const int m0 = blockIdx.y * MT;
    const int ca = min(col0, n - 1), cb = min(col0 + 1, n - 1);
    const int nbk = k / 32;
    const uint4* qa = reinterpret_cast<const uint4*>(quants) + static_cast<size_t>(ca) * (k / 16);
    const uint4* qb = reinterpret_cast<const uint4*>(quants) + static_cast<size_t>(cb) * (k / 16);

    float2 acc[MT];
#pragma unroll
    for (int r = 0; r < MT; ++r) acc[r] = make_float2(0.0f, 0.0f);

    for (int kc = 0; kc < k; kc += kKC) {
        const int kn = min(kKC, k - kc);
        __syncthreads();
        for (int e = threadIdx.x; e < kn * MS; e += kThreads) {
            const int t = e / MS, r = e % MS;
            xs[t][r] = (r < MT) ? x[static_cast<size_t>(min(m0 + r, m - 1)) * k + kc + t] : 0.0f;
        }
        __syncthreads();
        const int b0 = kc / 32, nbl = kn / 32;
        uint4 na0 = __ldg(qa + 2 * b0), na1 = __ldg(qa + 2 * b0 + 1);
        uint4 nb0 = __ldg(qb + 2 * b0), nb1 = __ldg(qb + 2 * b0 + 1);
        for (int bl = 0; bl < nbl; ++bl) {
            const int b = b0 + bl;
            const uint4 a0 = na0, a1 = na1, c0 = nb0, c1 = nb1;
            if (bl + 1 < nbl) {
                na0 = __ldg(qa + 2 * b + 2);
                na1 = __ldg(qa + 2 * b + 3);
                nb0 = __ldg(qb + 2 * b + 2);
                nb1 = __ldg(qb + 2 * b + 3);
            }
            const uint32_t wa[8] = {a0.x ^ 0x80808080u, a0.y ^ 0x80808080u, a0.z ^ 0x80808080u, a0.w ^ 0x80808080u,
                                    a1.x ^ 0x80808080u, a1.y ^ 0x80808080u, a1.z ^ 0x80808080u, a1.w ^ 0x80808080u};
            const uint32_t wb[8] = {c0.x ^ 0x80808080u, c0.y ^ 0x80808080u, c0.z ^ 0x80808080u, c0.w ^ 0x80808080u,
                                    c1.x ^ 0x80808080u, c1.y ^ 0x80808080u, c1.z ^ 0x80808080u, c1.w ^ 0x80808080u};
            float2 bs[MT];
#pragma unroll
            for (int r = 0; r < MT; ++r) bs[r] = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int t = 0; t < 32; ++t) {
                const float2 qq = make_float2(q_of(wa[t >> 2], t & 3), q_of(wb[t >> 2], t & 3));
                const float* xr = &xs[bl * 32 + t][0];
#pragma unroll
                for (int r = 0; r < MT; r += 4) {
                    const float4 xv = *reinterpret_cast<const float4*>(xr + r);
                    bs[r] = fadd2(bs[r], mul_pair(xv.x, qq));
                    if (r + 1 < MT) bs[r + 1] = fadd2(bs[r + 1], mul_pair(xv.y, qq));
                    if (r + 2 < MT) bs[r + 2] = fadd2(bs[r + 2], mul_pair(xv.z, qq));
                    if (r + 3 < MT) bs[r + 3] = fadd2(bs[r + 3], mul_pair(xv.w, qq));
                }
            }
            const float2 sc = make_float2(__ldg(scales + static_cast<size_t>(ca) * nbk + b),
                                          __ldg(scales + static_cast<size_t>(cb) * nbk + b));
#pragma unroll
            for (int r = 0; r < MT; ++r)
                acc[r] = fadd2(acc[r], make_float2(__fmul_rn(sc.x, bs[r].x), __fmul_rn(sc.y, bs[r].y)));
        }
    }
    if (col0 < n) {
#pragma unroll
        for (int r = 0; r < MT; ++r) {
            const int row = m0 + r;
            if (row < m) {
                y[static_cast<size_t>(row) * n + col0] = acc[r].x;
                if (col0 + 1 < n) y[static_cast<size_t>(row) * n + col0 + 1] = acc[r].y;
            }
        }
    }
}

template <int MT>
cudaError_t launch_mt(const float* x, const uint32_t* q, const float* s, float* y, int m, int k, int n,
                      cudaStream_t st) {
    const dim3 grid((n + 2 * kThreads - 1) / (2 * kThreads), (m + MT - 1) / MT);
    block_q8_kernel<MT><<<grid, kThreads, 0, st>>>(x, q, s, y, m, k, n);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_block_q8(const float* x, const uint32_t* quants, const float* scales, float* y, int m, int k,
                            int n, cudaStream_t s) {
    if (m <= 1) return launch_mt<1>(x, quants, scales, y, m, k, n, s);
    if (m <= 2) return launch_mt<2>(x, quants, scales, y, m, k, n, s);
    if (m <= 4) return launch_mt<4>(x, quants, scales, y, m, k, n, s);
    if (m <= 8) return launch_mt<8>(x, quants, scales, y, m, k, n, s);
    return launch_mt<16>(x, quants, scales, y, m, k, n, s);
}

}  // namespace gq
