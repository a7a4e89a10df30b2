// Block-quantized weights times f32 activations on sm_103a (web-xpu-ops README: the op table rows
// matvecQ8 / matmulQ8 and matvecQ4G128 / matmulQ4G128, and "The q4 format").
//   8 bits: code k of row n is byte k % 4 of word n * K/4 + k/4 (least-significant first, signed);
//           y[t, n] = scale[n] * sum_k q(n, k) * x[t, k] -- the row scale applied once at the end.
//   4 bits: code k of row n is nibble k % 8 of word n * K/8 + k/8 (least-significant first, 4-bit
//           two's complement); y[t, n] = sum_g scale[n, g] * sum_{k in g} q(n, k) * x[t, k] over
//           groups of 128 columns.
// The page fixes no float order, so results are checked against the exact value within an error
// bound of each kernel's own order.
//
// Codes become floats exactly: a biased code (byte ^ 0x80, or nibble ^ 8) is placed in the low bits
// of 2^23's bit pattern by a byte permute, and one subtraction removes 2^23 plus the bias.
//
// GEMV (T <= 4 tokens): a thread block covers 32/T rows, 8 at a time; its eight warps take the
// 512-column chunks of K in turn (chunk c to warp c % 8), each lane 16 consecutive columns of a
// chunk, so a warp's load of one row is 512 (8-bit) or 256 (4-bit) contiguous bytes.  Per (row,
// token) a lane keeps the even- and odd-column sums as one f32 pair; after the chunks the lanes
// are reduced by halving exchanges and the eight warps' totals are added in a fixed tree.
//
// GEMM (T > 4): a thread block computes 128 rows x 128 tokens, K staged 32 columns at a time.  The
// codes are turned into floats (times the group scale for 4 bits) into shared memory once per
// stage, and each thread accumulates an 8 x 8 block of outputs from outer products.
#include "gq_internal.cuh"

namespace gq {
namespace {

// Exact float of a signed byte / 4-bit code, from the biased field in the low byte.
__device__ __forceinline__ float biased_byte_to_f32(uint32_t biased_word, int j) {
    return __fsub_rn(__uint_as_float(__byte_perm(biased_word, 0x4B000000u, 0x7440 + j)), 8388736.0f);   // 2^23 + 128
}
__device__ __forceinline__ float biased_nibble_to_f32(uint32_t biased_bytes, int j) {
    return __fsub_rn(__uint_as_float(__byte_perm(biased_bytes, 0x4B000000u, 0x7440 + j)), 8388616.0f);   // 2^23 + 8
}

// The 16 codes of one lane's slice, in column order.
template <int BITS>
__device__ __forceinline__ void decode16(const uint32_t (&wd)[BITS == 8 ? 4 : 2], float (&cf)[16]) {
    if constexpr (BITS == 8) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t b = wd[i] ^ 0x80808080u;
#pragma unroll
            for (int j = 0; j < 4; ++j) cf[4 * i + j] = biased_byte_to_f32(b, j);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const uint32_t ev = (wd[i] & 0x0F0F0F0Fu) ^ 0x08080808u;          // nibbles 0, 2, 4, 6
            const uint32_t od = ((wd[i] >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;   // nibbles 1, 3, 5, 7
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                cf[8 * i + 2 * j] = biased_nibble_to_f32(ev, j);
                cf[8 * i + 2 * j + 1] = biased_nibble_to_f32(od, j);
            }
        }
    }
}

constexpr int kGvWarps = 8;
constexpr int kChunk = 512;                       // columns per warp step (16 per lane)

__device__ __forceinline__ float2 fsub2(float2 a, float2 b) {
    return fadd2(a, make_float2(-b.x, -b.y));     // negation is exact
}

// The 16 codes of one lane's slice as 8 float pairs (codes 2i, 2i+1), exact.
template <int BITS>
__device__ __forceinline__ void decode16x2(const uint32_t (&wd)[BITS == 8 ? 4 : 2], float2 (&cf)[8]) {
    if constexpr (BITS == 8) {
        const float2 bias = make_float2(8388736.0f, 8388736.0f);             // 2^23 + 128
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t b = wd[i] ^ 0x80808080u;
            cf[2 * i] = fsub2(make_float2(__uint_as_float(__byte_perm(b, 0x4B000000u, 0x7440)),
                                          __uint_as_float(__byte_perm(b, 0x4B000000u, 0x7441))), bias);
            cf[2 * i + 1] = fsub2(make_float2(__uint_as_float(__byte_perm(b, 0x4B000000u, 0x7442)),
                                              __uint_as_float(__byte_perm(b, 0x4B000000u, 0x7443))), bias);
        }
    } else {
        const float2 bias = make_float2(8388616.0f, 8388616.0f);             // 2^23 + 8
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const uint32_t ev = (wd[i] & 0x0F0F0F0Fu) ^ 0x08080808u;          // nibbles 0, 2, 4, 6
            const uint32_t od = ((wd[i] >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;   // nibbles 1, 3, 5, 7
#pragma unroll
            for (int j = 0; j < 4; ++j)
                cf[4 * i + j] = fsub2(make_float2(__uint_as_float(__byte_perm(ev, 0x4B000000u, 0x7440 + j)),
                                                  __uint_as_float(__byte_perm(od, 0x4B000000u, 0x7440 + j))), bias);
        }
    }
}

// Launched as a programmatic dependent: a warp's first weight loads are issued before the wait for
// the preceding grids; the activations are read and the outputs written after it.
// GEMV: 32/T rows per thread block, taken 8 rows at a time; warp w takes the 512-column chunks
// w, w + 8, ... of K.  A lane keeps two partial sums per (row, token) -- even and odd columns of
// its 16 -- as one f32 pair (fma.f32x2), adds them at the end of its chunks, and the lanes are
// then reduced by halving exchanges (lane l ends with value (l >> (5 - log2 V)) of the V = 8T).
template <int BITS, int T>
__global__ void __launch_bounds__(kGvWarps * 32, T == 1 ? 3 : 1)   // one token: 3 blocks per SM, one wave
wq_gemv_kernel(const uint32_t* __restrict__ w, const float* __restrict__ scale, const float* __restrict__ x,
               float* __restrict__ y, int N, int K, int Tn) {
    constexpr int R = 32 / T;                     // rows per thread block
    constexpr int V = 8 * T;                      // values per lane per row batch
    constexpr int WPL = BITS == 8 ? 4 : 2;        // words per lane per chunk
    __shared__ float part[kGvWarps][R * T];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * R;
    const size_t wpr = static_cast<size_t>(K) * BITS / 32;   // words per row
    const int G = (K + 127) / 128;
    const int nchunks = (K + kChunk - 1) / kChunk;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    bool waited = false;

#pragma unroll
    for (int rb = 0; rb < R; rb += 8) {
        float2 acc[8][T];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int u = 0; u < T; ++u) acc[i][u] = make_float2(0.0f, 0.0f);
        for (int c = warp; c < nchunks; c += kGvWarps) {
            const int k0 = c * kChunk + 16 * lane;
            if (k0 < K) {                         // K % 32 == 0: a live lane has all 16 columns
                uint32_t wd[8][WPL];
                float sc[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int n = min(n0 + rb + i, N - 1);        // past-the-end rows: computed, not stored
                    const uint32_t* p = w + static_cast<size_t>(n) * wpr + static_cast<size_t>(k0) * BITS / 32;
                    if constexpr (BITS == 8) {
                        const uint4 a = __ldg(reinterpret_cast<const uint4*>(p));
                        wd[i][0] = a.x; wd[i][1] = a.y; wd[i][2] = a.z; wd[i][3] = a.w;
                    } else {
                        const uint2 a = __ldg(reinterpret_cast<const uint2*>(p));
                        wd[i][0] = a.x; wd[i][1] = a.y;
                        sc[i] = __ldg(scale + static_cast<size_t>(n) * G + k0 / 128);
                    }
                }
                if (!waited) {
                    asm volatile("griddepcontrol.wait;" ::: "memory");   // the preceding grids are done
                    waited = true;
                }
                float2 xv[T][8];
#pragma unroll
                for (int u = 0; u < T; ++u) {
                    // tokens past Tn (a 3-token call through the 4-token kernel) repeat the last one
                    const float4* xp = reinterpret_cast<const float4*>(x + static_cast<size_t>(min(u, Tn - 1)) * K + k0);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float4 a = __ldg(xp + q);
                        xv[u][2 * q] = make_float2(a.x, a.y);
                        xv[u][2 * q + 1] = make_float2(a.z, a.w);
                    }
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    float2 cf[8];
                    decode16x2<BITS>(wd[i], cf);
#pragma unroll
                    for (int u = 0; u < T; ++u) {
                        if constexpr (BITS == 8) {
#pragma unroll
                            for (int j = 0; j < 8; ++j) acc[i][u] = ffma2(cf[j], xv[u][j], acc[i][u]);
                        } else {
                            float2 p = fmul2(cf[0], xv[u][0]);
#pragma unroll
                            for (int j = 1; j < 8; ++j) p = ffma2(cf[j], xv[u][j], p);
                            // one sum per (row, token) for 4 bits: the even/odd pair is added first
                            acc[i][u].x = __fmaf_rn(sc[i], __fadd_rn(p.x, p.y), acc[i][u].x);
                        }
                    }
                }
            }
        }
        float v[V];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int u = 0; u < T; ++u) v[i * T + u] = __fadd_rn(acc[i][u].x, acc[i][u].y);
        // halving exchanges over lane bits 4, 3, ... until one value is left, then plain butterflies
#pragma unroll
        for (int h = V / 2, m = 16; h >= 1; h >>= 1, m >>= 1) {
            const bool hi = (lane & m) != 0;
#pragma unroll
            for (int j = 0; j < h; ++j) {
                const float send = hi ? v[j] : v[j + h];
                const float keep = hi ? v[j + h] : v[j];
                v[j] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, m));
            }
        }
#pragma unroll
        for (int m = 16 / V; m >= 1; m >>= 1) v[0] = __fadd_rn(v[0], __shfl_xor_sync(0xffffffffu, v[0], m));
        const int idx = lane / (32 / V);          // (row i, token u) = (idx / T, idx % T)
        if (lane % (32 / V) == 0) part[warp][rb * T + idx] = v[0];
    }
    if (!waited) asm volatile("griddepcontrol.wait;" ::: "memory");   // warps with no chunk
    __syncthreads();
    for (int e = threadIdx.x; e < R * T; e += blockDim.x) {
        const float tot = __fadd_rn(__fadd_rn(__fadd_rn(part[0][e], part[1][e]), __fadd_rn(part[2][e], part[3][e])),
                                    __fadd_rn(__fadd_rn(part[4][e], part[5][e]), __fadd_rn(part[6][e], part[7][e])));
        const int n = n0 + e / T, u = e % T;
        if (n < N && u < Tn) {
            const float out = (BITS == 8) ? __fmul_rn(__ldg(scale + n), tot) : tot;
            y[static_cast<size_t>(u) * N + n] = out;
        }
    }
}

// W4 GEMV for one token: the same bytes in flight per lane as the 8-bit kernel.  A lane takes 32
// consecutive columns (16 bytes) of a row, so a warp step covers 1024 columns; a thread block
// covers 48 rows in batches of 16, and warp w takes row half w >> 2 of each batch and the 1024-column chunks (w & 3), (w & 3) + 4, ... of K.  Per
// (row, chunk) a lane forms the 32-column sum as an even/odd f32 pair (16-term chains), adds the
// pair and folds it in with one fma by the group scale (32 columns lie in one 128-column group);
// then the halving exchanges, and a fixed tree of the four chunk phases' partials.
constexpr int kG4Chunk = 1024;
constexpr int kG4Rows = 48;                        // rows per thread block, three batches of 16
__global__ void __launch_bounds__(kGvWarps * 32, 2)   // two blocks per SM: 14,336 rows in one wave
wq4_gemv1_kernel(const uint32_t* __restrict__ w, const float* __restrict__ scale, const float* __restrict__ x,
                 float* __restrict__ y, int N, int K) {
    constexpr int R = kG4Rows;
    __shared__ float part[4][R];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int half = warp >> 2, phase = warp & 3;
    const int n0 = blockIdx.x * R;
    const size_t wpr = static_cast<size_t>(K) / 8;            // words per row
    const int G = (K + 127) / 128;
    const int nchunks = (K + kG4Chunk - 1) / kG4Chunk;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    bool waited = false;
#pragma unroll 1
    for (int rb = 0; rb < R; rb += 16) {
        const int r0 = rb + 8 * half;             // this warp's 8 rows: r0 .. r0 + 7
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
        for (int c = phase; c < nchunks; c += 4) {
            const int k0 = c * kG4Chunk + 32 * lane;
            if (k0 < K) {                         // K % 32 == 0: a live lane has all 32 columns
                uint32_t wd[8][4];
                float sc[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int n = min(n0 + r0 + i, N - 1);        // past-the-end rows: computed, not stored
                    const uint4 a = __ldg(reinterpret_cast<const uint4*>(w + static_cast<size_t>(n) * wpr + k0 / 8));
                    wd[i][0] = a.x; wd[i][1] = a.y; wd[i][2] = a.z; wd[i][3] = a.w;
                    sc[i] = __ldg(scale + static_cast<size_t>(n) * G + k0 / 128);
                }
                if (!waited) {
                    asm volatile("griddepcontrol.wait;" ::: "memory");   // the preceding grids are done
                    waited = true;
                }
                const float4* xp = reinterpret_cast<const float4*>(x + k0);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {  // columns 16 hh .. 16 hh + 15
                    float2 xv[8];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float4 a = __ldg(xp + 4 * hh + q);
                        xv[2 * q] = make_float2(a.x, a.y);
                        xv[2 * q + 1] = make_float2(a.z, a.w);
                    }
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const uint32_t wh[2] = {wd[i][2 * hh], wd[i][2 * hh + 1]};
                        float2 cf[8];
                        decode16x2<4>(wh, cf);
                        // the even/odd chains run on over the second 16 columns (the first
                        // half's pair is parked in the consumed code words)
                        float2 p = (hh == 0) ? fmul2(cf[0], xv[0])
                                             : ffma2(cf[0], xv[0], make_float2(__uint_as_float(wd[i][0]),
                                                                               __uint_as_float(wd[i][1])));
#pragma unroll
                        for (int j = 1; j < 8; ++j) p = ffma2(cf[j], xv[j], p);
                        if (hh == 0) {
                            wd[i][0] = __float_as_uint(p.x);
                            wd[i][1] = __float_as_uint(p.y);
                        } else {
                            acc[i] = __fmaf_rn(sc[i], __fadd_rn(p.x, p.y), acc[i]);
                        }
                    }
                }
            }
        }
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = acc[i];
        // halving exchanges over lane bits 4, 3, 2, then butterflies over bits 1, 0
#pragma unroll
        for (int h = 4, m = 16; h >= 1; h >>= 1, m >>= 1) {
            const bool hi = (lane & m) != 0;
#pragma unroll
            for (int j = 0; j < h; ++j) {
                const float send = hi ? v[j] : v[j + h];
                const float keep = hi ? v[j + h] : v[j];
                v[j] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, m));
            }
        }
#pragma unroll
        for (int m = 2; m >= 1; m >>= 1) v[0] = __fadd_rn(v[0], __shfl_xor_sync(0xffffffffu, v[0], m));
        if ((lane & 3) == 0) part[phase][r0 + (lane >> 2)] = v[0];
    }
    if (!waited) asm volatile("griddepcontrol.wait;" ::: "memory");   // warps with no chunk
    __syncthreads();
    if (threadIdx.x < R) {
        const int n = n0 + threadIdx.x;
        if (n < N)
            y[n] = __fadd_rn(__fadd_rn(part[0][threadIdx.x], part[1][threadIdx.x]),
                             __fadd_rn(part[2][threadIdx.x], part[3][threadIdx.x]));
    }
}

// ------------------------------------------------------------------------------------- GEMM

constexpr int kGmN = 128, kGmT = 128, kGmK = 32;  // tile: rows x tokens x columns per stage
constexpr int kGmPad = 4;                         // row padding of the [k][n] / [k][t] stage arrays

template <int BITS>
__global__ void __launch_bounds__(256)
wq_gemm_kernel(const uint32_t* __restrict__ w, const float* __restrict__ scale, const float* __restrict__ x,
               float* __restrict__ y, int T, int N, int K) {
    __shared__ __align__(16) float Ws[kGmK][kGmN + kGmPad];
    __shared__ __align__(16) float Xs[kGmK][kGmT + kGmPad];
    const int tid = threadIdx.x;
    // 16 x 16 threads; thread (tx, ty) owns rows 4tx..4tx+3 and 64+4tx..+3, tokens 4ty.. and 64+4ty..
    // (a quarter-warp's 16-byte reads then cover 128 contiguous bytes)
    const int tx = tid & 15, ty = tid >> 4;
    const int n0 = blockIdx.x * kGmN, t0 = blockIdx.y * kGmT;
    const size_t wpr = static_cast<size_t>(K) * BITS / 32;
    const int G = (K + 127) / 128;
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;

    for (int k0 = 0; k0 < K; k0 += kGmK) {
        __syncthreads();                          // the previous stage is consumed
        // weights: 128 rows x 32 codes; 8 bits: thread -> (row tid/2, 16 codes); 4 bits: (row tid/2, 16 codes)
        {
            const int r = tid >> 1, half = tid & 1;
            const int n = min(n0 + r, N - 1);
            const uint32_t* p = w + static_cast<size_t>(n) * wpr + static_cast<size_t>(k0 + 16 * half) * BITS / 32;
            uint32_t wd[BITS == 8 ? 4 : 2];
            if constexpr (BITS == 8) {
                const uint4 a = __ldg(reinterpret_cast<const uint4*>(p));
                wd[0] = a.x; wd[1] = a.y; wd[2] = a.z; wd[3] = a.w;
            } else {
                const uint2 a = __ldg(reinterpret_cast<const uint2*>(p));
                wd[0] = a.x; wd[1] = a.y;
            }
            float cf[16];
            decode16<BITS>(wd, cf);
            if constexpr (BITS == 4) {
                const float sc = __ldg(scale + static_cast<size_t>(n) * G + k0 / 128);
#pragma unroll
                for (int j = 0; j < 16; ++j) cf[j] = __fmul_rn(cf[j], sc);
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) Ws[16 * half + j][r] = cf[j];
        }
        // activations: 128 tokens x 32 columns; thread -> (token tid/2, 16 columns)
        {
            const int tt = tid >> 1, half = tid & 1;
            const int t = min(t0 + tt, T - 1);
            const float4* xp = reinterpret_cast<const float4*>(x + static_cast<size_t>(t) * K + k0 + 16 * half);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 a = __ldg(xp + q);
                Xs[16 * half + 4 * q][tt] = a.x;
                Xs[16 * half + 4 * q + 1][tt] = a.y;
                Xs[16 * half + 4 * q + 2][tt] = a.z;
                Xs[16 * half + 4 * q + 3][tt] = a.w;
            }
        }
        __syncthreads();
#pragma unroll 4
        for (int kk = 0; kk < kGmK; ++kk) {
            const float4 a0 = *reinterpret_cast<const float4*>(&Ws[kk][4 * tx]);
            const float4 a1 = *reinterpret_cast<const float4*>(&Ws[kk][64 + 4 * tx]);
            const float4 b0 = *reinterpret_cast<const float4*>(&Xs[kk][4 * ty]);
            const float4 b1 = *reinterpret_cast<const float4*>(&Xs[kk][64 + 4 * ty]);
            const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = __fmaf_rn(a[i], b[j], acc[i][j]);
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int n = n0 + (i < 4 ? 4 * tx + i : 64 + 4 * tx + i - 4);
        if (n >= N) continue;
        const float sc = (BITS == 8) ? __ldg(scale + n) : 1.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int t = t0 + (j < 4 ? 4 * ty + j : 64 + 4 * ty + j - 4);
            if (t < T) y[static_cast<size_t>(t) * N + n] = (BITS == 8) ? __fmul_rn(sc, acc[i][j]) : acc[i][j];
        }
    }
}

template <int BITS, int T>
cudaError_t launch_gemv(const uint32_t* w, const float* scale, const float* x, float* y, int N, int K, int Tn,
                        cudaStream_t s) {
    constexpr int R = 32 / T;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((N + R - 1) / R);
    cfg.blockDim = dim3(kGvWarps * 32);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, wq_gemv_kernel<BITS, T>, w, scale, x, y, N, K, Tn);
}

template <int BITS>
cudaError_t launch_bits(const uint32_t* w, const float* scale, const float* x, float* y, int T, int N, int K,
                        cudaStream_t s) {
    if (T == 1 && BITS == 4) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((N + kG4Rows - 1) / kG4Rows);
        cfg.blockDim = dim3(kGvWarps * 32);
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, wq4_gemv1_kernel, w, scale, x, y, N, K);
    }
    if (T == 1) return launch_gemv<BITS, 1>(w, scale, x, y, N, K, T, s);
    if (T == 2) return launch_gemv<BITS, 2>(w, scale, x, y, N, K, T, s);
    if (T <= 4) return launch_gemv<BITS, 4>(w, scale, x, y, N, K, T, s);
    const dim3 grid((N + kGmN - 1) / kGmN, (T + kGmT - 1) / kGmT);
    wq_gemm_kernel<BITS><<<grid, 256, 0, s>>>(w, scale, x, y, T, N, K);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_wq(int bits, const uint32_t* w, const float* scale, const float* x, float* y, int T, int N, int K,
                      cudaStream_t s) {
    return bits == 8 ? launch_bits<8>(w, scale, x, y, T, N, K, s) : launch_bits<4>(w, scale, x, y, T, N, K, s);
}

}  // namespace gq
