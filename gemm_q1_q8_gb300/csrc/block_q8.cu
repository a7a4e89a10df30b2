// block_q8_matmul_nt on sm_103a (kopitiam-gpu block_q8_matmul_nt.wgsl): y = x . w^T with int8
// weights packed four per u32 (little-endian, sign-extended) and one f32 scale per 32-block.
// Order, bit for bit: per (row, col), block b ascending: block_sum = 0; block_sum = block_sum +
// x*q for t = 0..31 (a rounded multiply, then a rounded add); acc = acc + scale*block_sum.
//
// The block sums of a column are independent of one another; only the final `acc` chain runs in
// block order.  For few activation rows (m <= 4) a thread block covers 32 columns: its warps take the 32-blocks in turn (warp w
// the blocks w, w+W, ...), each lane one column, so a warp's activation reads are broadcasts and
// each lane reads its column's 32 bytes of the block directly (the next block's bytes load while
// the current one is summed).  The scaled block sums (scale*block_sum, rounded) go to shared
// memory for a pass of blocks, then the thread that owns a (row, column) adds them into its acc in
// block order.  The activations sit transposed in shared memory (one broadcast load feeds up to four
// rows), staged once for up to 64 KB of them; an int8 becomes an exact f32 as bits 0x4B0000xx
// (2^23 + q + 128) minus 2^23 + 128.  Pairs of rows share packed f32x2 adds (each lane one IEEE
// operation); the products stay scalar on purpose: ptxas contracts a packed mul.rn.f32x2 that
// feeds a packed add.rn.f32x2 into one fused fma.rn.f32x2 (observed on sm_103a), which would
// change the rounding of every step; a scalar mul.rn is never contracted.
#include "gq_internal.cuh"

namespace gq {
namespace {

constexpr int kColsPerCta = 32;           // one column per lane
// warps per thread block: 4 for small m (16 blocks per SM, so n = 49152 fits in one wave), 8 for
// m >= 8 (more rows per lane: fewer, fuller blocks)
template <int MT>
__host__ __device__ constexpr int warps_of() { return MT >= 8 ? 8 : 4; }
constexpr int kXBytes = 64 * 1024;        // activations staged at once (transposed)
constexpr float kQBias = 8388736.0f;      // 2^23 + 128

template <int MT>
__host__ __device__ constexpr int x_stride() { return MT; }   // rows of a staged activation column

// blocks per pass: the scaled block sums of a pass (pass x MT x 32 floats) stay within 32 KB
template <int MT>
__host__ __device__ constexpr int pass_blocks() { return MT <= 4 ? 64 : (MT <= 8 ? 32 : 16); }

// k values staged per activation pass: a multiple of 32 * pass_blocks within kXBytes
template <int MT>
__host__ __device__ constexpr int x_span() {
    return kXBytes / (x_stride<MT>() * 4) / (32 * pass_blocks<MT>()) * (32 * pass_blocks<MT>());
}

template <int MT>
size_t bq8_smem(int k) {
    const int span = k < x_span<MT>() ? k : x_span<MT>();   // k is a multiple of 32
    return static_cast<size_t>(span) * x_stride<MT>() * 4 +
           static_cast<size_t>(pass_blocks<MT>()) * MT * kColsPerCta * 4;
}

// element j (0..3) of a word already XORed with 0x80808080, as an exact float
__device__ __forceinline__ float q_of(uint32_t u, int j) {
    return __int_as_float(static_cast<int>(__byte_perm(u, 0x4B000000u, 0x7540u | j))) - kQBias;
}

// block_sum[r] += x[r] * q for the MT rows (rounded product, then rounded add; pairs of rows
// through one packed add)
template <int MT>
__device__ __forceinline__ void accumulate_rows(float (&bs)[MT], const float* xr, float q) {
    if constexpr (MT == 1) {
        bs[0] = __fadd_rn(bs[0], __fmul_rn(xr[0], q));
    } else if constexpr (MT == 2) {
        const float2 xv = *reinterpret_cast<const float2*>(xr);
        const float2 v = fadd2(make_float2(bs[0], bs[1]), make_float2(__fmul_rn(xv.x, q), __fmul_rn(xv.y, q)));
        bs[0] = v.x;
        bs[1] = v.y;
    } else {
#pragma unroll
        for (int r = 0; r < MT; r += 4) {
            const float4 xv = *reinterpret_cast<const float4*>(xr + r);
            const float2 lo =
                fadd2(make_float2(bs[r], bs[r + 1]), make_float2(__fmul_rn(xv.x, q), __fmul_rn(xv.y, q)));
            bs[r] = lo.x;
            bs[r + 1] = lo.y;
            if (r + 2 < MT) {
                const float2 hi =
                    fadd2(make_float2(bs[r + 2], bs[r + 3]), make_float2(__fmul_rn(xv.z, q), __fmul_rn(xv.w, q)));
                bs[r + 2] = hi.x;
                bs[r + 3] = hi.y;
            }
        }
    }
}

template <int MT>
__global__ void __launch_bounds__(warps_of<MT>() * 32)
block_q8_kernel(const float* __restrict__ x, const uint32_t* __restrict__ quants, const float* __restrict__ scales,
                float* __restrict__ y, int m, int k, int n) {
    constexpr int MS = x_stride<MT>();
    constexpr int PB = pass_blocks<MT>();
    constexpr int kWarps = warps_of<MT>();
    constexpr int kThreads = kWarps * 32;
    constexpr int kOwned = (MT * kColsPerCta + kThreads - 1) / kThreads;   // (row, column) pairs per thread
    extern __shared__ __align__(16) float smem_f[];
    const int span = k < x_span<MT>() ? k : x_span<MT>();   // all of k, or whole passes of blocks
    float* xs = smem_f;                              // [span][MS]
    float* ps = smem_f + span * MS;                  // [PB][MT][32] scaled block sums of a pass
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int col0 = blockIdx.x * kColsPerCta;
    const int m0 = blockIdx.y * MT;
    const int nbk = k / 32;
    const int cl = min(col0 + lane, n - 1);          // past-the-end columns compute column n-1, store nothing
    const uint4* qc = reinterpret_cast<const uint4*>(quants) + static_cast<size_t>(cl) * (k / 16);
    const float* sc = scales + static_cast<size_t>(cl) * nbk;

    float acc[kOwned];
#pragma unroll
    for (int o = 0; o < kOwned; ++o) acc[o] = 0.0f;

    for (int pb0 = 0; pb0 < nbk; pb0 += PB) {
        const int npb = min(PB, nbk - pb0);
        if ((pb0 * 32) % span == 0) {                // the next pass of activations, transposed
            __syncthreads();
            const int kc = pb0 * 32, kx = min(span, k - kc);
            for (int e = threadIdx.x; e < kx * MS; e += kThreads) {
                const int tt = e / MS, r = e % MS;
                xs[tt * MS + r] = (r < MT) ? x[static_cast<size_t>(min(m0 + r, m - 1)) * k + kc + tt] : 0.0f;
            }
            __syncthreads();
        }
        const float* xp = xs + ((pb0 * 32) % span) * MS;
        // this warp's blocks of the pass: pb0 + warp, pb0 + warp + kWarps, ...; the next two are
        // in flight while one is summed
        uint4 n0 = make_uint4(0u, 0u, 0u, 0u), n1 = n0, f0 = n0, f1 = n0;
        float nsc = 0.0f, fsc = 0.0f;
        if (warp < npb) {
            n0 = __ldg(qc + 2 * (pb0 + warp));
            n1 = __ldg(qc + 2 * (pb0 + warp) + 1);
            nsc = __ldg(sc + pb0 + warp);
        }
        if (warp + kWarps < npb) {
            f0 = __ldg(qc + 2 * (pb0 + warp + kWarps));
            f1 = __ldg(qc + 2 * (pb0 + warp + kWarps) + 1);
            fsc = __ldg(sc + pb0 + warp + kWarps);
        }
        for (int bl = warp; bl < npb; bl += kWarps) {
            const uint4 w0 = n0, w1 = n1;
            const float s = nsc;
            n0 = f0;
            n1 = f1;
            nsc = fsc;
            if (bl + 2 * kWarps < npb) {
                f0 = __ldg(qc + 2 * (pb0 + bl + 2 * kWarps));
                f1 = __ldg(qc + 2 * (pb0 + bl + 2 * kWarps) + 1);
                fsc = __ldg(sc + pb0 + bl + 2 * kWarps);
            }
            const uint32_t wq[8] = {w0.x ^ 0x80808080u, w0.y ^ 0x80808080u, w0.z ^ 0x80808080u,
                                    w0.w ^ 0x80808080u, w1.x ^ 0x80808080u, w1.y ^ 0x80808080u,
                                    w1.z ^ 0x80808080u, w1.w ^ 0x80808080u};
            float bs[MT];
#pragma unroll
            for (int r = 0; r < MT; ++r) bs[r] = 0.0f;
            const float* xb = xp + bl * 32 * MS;
            if constexpr (MT == 1) {
                // one broadcast float4 per four activations
#pragma unroll
                for (int t4 = 0; t4 < 8; ++t4) {
                    const float4 xv = *reinterpret_cast<const float4*>(xb + 4 * t4);
                    bs[0] = __fadd_rn(bs[0], __fmul_rn(xv.x, q_of(wq[t4], 0)));
                    bs[0] = __fadd_rn(bs[0], __fmul_rn(xv.y, q_of(wq[t4], 1)));
                    bs[0] = __fadd_rn(bs[0], __fmul_rn(xv.z, q_of(wq[t4], 2)));
                    bs[0] = __fadd_rn(bs[0], __fmul_rn(xv.w, q_of(wq[t4], 3)));
                }
            } else {
#pragma unroll
                for (int tt = 0; tt < 32; ++tt) accumulate_rows<MT>(bs, xb + tt * MS, q_of(wq[tt >> 2], tt & 3));
            }
#pragma unroll
            for (int r = 0; r < MT; ++r) ps[(bl * MT + r) * kColsPerCta + lane] = __fmul_rn(s, bs[r]);
        }
        __syncthreads();
        // acc = acc + scale*block_sum, block by block in order, for the owned (row, column) pairs
#pragma unroll
        for (int o = 0; o < kOwned; ++o) {
            const int pr = threadIdx.x + o * kThreads;
            if (pr < MT * kColsPerCta) {
                const int r = pr / kColsPerCta, c = pr % kColsPerCta;
                float a = acc[o];
                for (int bl = 0; bl < npb; ++bl) a = __fadd_rn(a, ps[(bl * MT + r) * kColsPerCta + c]);
                acc[o] = a;
            }
        }
        __syncthreads();                              // the pass's sums are read before the next pass
    }
#pragma unroll
    for (int o = 0; o < kOwned; ++o) {
        const int pr = threadIdx.x + o * kThreads;
        if (pr < MT * kColsPerCta) {
            const int r = pr / kColsPerCta, c = pr % kColsPerCta;
            const int row = m0 + r, col = col0 + c;
            if (row < m && col < n) y[static_cast<size_t>(row) * n + col] = acc[o];
        }
    }
}

// One or two activation rows: a lane takes a whole 32-block of a weight row (its 32 codes are 32
// contiguous bytes, so a warp's two 16-byte loads per row cover 1 KB of the row, coalesced), keeps
// the block's activations in registers for every row, and runs the block sum in order; the warp's
// rows are summed side by side (one independent chain per row).  The rounded products
// scale*block_sum go through shared memory to lane r, which adds row r's blocks in order.  Blocks
// beyond 32 per row are taken 32 at a time, the owner's acc carrying on across them.
// Launched as a programmatic dependent: the first weight rows are requested before the wait for
// the preceding grids, the activations read and the outputs written after it.
constexpr int kRwWarps = 8;

// rows per warp: one independent block-sum chain each.  Seven for one token: 126 registers, two
// thread blocks per SM, and for n = 49152 about 2.9 waves of warps (eight rows: 2.5 waves, whose
// half-empty last wave cost ~8%)
template <int MT>
__host__ __device__ constexpr int rw_rows() { return MT == 1 ? 7 : 4; }

template <int MT>
__global__ void __launch_bounds__(kRwWarps * 32)
block_q8_rowwarp_kernel(const float* __restrict__ x, const uint32_t* __restrict__ quants,
                        const float* __restrict__ scales, float* __restrict__ y, int m, int k, int n) {
    constexpr int R = rw_rows<MT>();
    __shared__ float ps[kRwWarps][R][33];           // a warp's rounded block products, odd stride
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nbk = k / 32;
    const int row0 = (blockIdx.x * kRwWarps + warp) * R;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (row0 >= n) return;                           // whole warps only: no block-wide barrier below
    float accs[MT];                                  // lane r < R: row row0 + r
#pragma unroll
    for (int u = 0; u < MT; ++u) accs[u] = 0.0f;
    for (int c0 = 0; c0 < nbk; c0 += 32) {
        const int b = c0 + lane;
        const bool live = b < nbk;
        uint32_t wq[R][8];
        float sc[R];
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const int row = min(row0 + i, n - 1);    // past-the-end rows: computed, not stored
            const uint4* qp = reinterpret_cast<const uint4*>(quants) + static_cast<size_t>(row) * (k / 16) +
                              2 * static_cast<size_t>(live ? b : 0);
            const uint4 w0 = __ldg(qp), w1 = __ldg(qp + 1);
            wq[i][0] = w0.x ^ 0x80808080u; wq[i][1] = w0.y ^ 0x80808080u; wq[i][2] = w0.z ^ 0x80808080u;
            wq[i][3] = w0.w ^ 0x80808080u; wq[i][4] = w1.x ^ 0x80808080u; wq[i][5] = w1.y ^ 0x80808080u;
            wq[i][6] = w1.z ^ 0x80808080u; wq[i][7] = w1.w ^ 0x80808080u;
            sc[i] = __ldg(scales + static_cast<size_t>(row) * nbk + (live ? b : 0));
        }
        if (c0 == 0) asm volatile("griddepcontrol.wait;" ::: "memory");   // the preceding grids are done
        // the block's activations for the MT tokens
        float xv[MT][32];
#pragma unroll
        for (int u = 0; u < MT; ++u) {
            const float4* xp = reinterpret_cast<const float4*>(x + static_cast<size_t>(u < m ? u : m - 1) * k +
                                                               static_cast<size_t>(live ? b : 0) * 32);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
                const float4 a = __ldg(xp + q4);
                xv[u][4 * q4] = a.x; xv[u][4 * q4 + 1] = a.y; xv[u][4 * q4 + 2] = a.z; xv[u][4 * q4 + 3] = a.w;
            }
        }
        float bs[R][MT];
#pragma unroll
        for (int i = 0; i < R; ++i)
#pragma unroll
            for (int u = 0; u < MT; ++u) bs[i][u] = 0.0f;
#pragma unroll
        for (int t = 0; t < 32; t += 2) {
#pragma unroll
            for (int i = 0; i < R; ++i) {
                // two codes at once: their biased floats, minus the bias in one packed (exact) subtraction
                const uint32_t wv = wq[i][t >> 2];
                const float2 q2 = fadd2(make_float2(__int_as_float(static_cast<int>(__byte_perm(wv, 0x4B000000u, 0x7540u | (t & 3)))),
                                                    __int_as_float(static_cast<int>(__byte_perm(wv, 0x4B000000u, 0x7540u | ((t & 3) + 1))))),
                                        make_float2(-kQBias, -kQBias));
#pragma unroll
                for (int u = 0; u < MT; ++u) {
                    bs[i][u] = __fadd_rn(bs[i][u], __fmul_rn(xv[u][t], q2.x));
                    bs[i][u] = __fadd_rn(bs[i][u], __fmul_rn(xv[u][t + 1], q2.y));
                }
            }
        }
        // per token: the rounded products to shared memory, lane r adds row r's in block order
#pragma unroll
        for (int u = 0; u < MT; ++u) {
#pragma unroll
            for (int i = 0; i < R; ++i) ps[warp][i][lane] = __fmul_rn(sc[i], bs[i][u]);
            __syncwarp();
            if (lane < R) {
                const int nb = min(32, nbk - c0);
                float a = accs[u];
                for (int j = 0; j < nb; ++j) a = __fadd_rn(a, ps[warp][lane][j]);
                accs[u] = a;
            }
            __syncwarp();
        }
    }
    if (lane < R && row0 + lane < n) {
#pragma unroll
        for (int u = 0; u < MT; ++u)
            if (u < m) y[static_cast<size_t>(u) * n + row0 + lane] = accs[u];
    }
}

// Many activation rows (m >= 8): each thread owns two weight columns and a tile of MT rows, the
// two columns' chains side by side (two scalar rounded products, then one packed add), so each
// broadcast activation load feeds two columns; the activation tile is staged transposed in passes
// of 256 values.
constexpr int kPairThreads = 256;
constexpr int kPairKC = 256;

// two rounded products, kept out of any contraction
__device__ __forceinline__ float2 pair_products(float a, float2 b) {
    return make_float2(__fmul_rn(a, b.x), __fmul_rn(a, b.y));
}

template <int MT>
__global__ void __launch_bounds__(kPairThreads)
block_q8_pair_kernel(const float* __restrict__ x, const uint32_t* __restrict__ quants, const float* __restrict__ scales,
                float* __restrict__ y, int m, int k, int n) {
    __shared__ __align__(16) float xs[kPairKC][MT < 4 ? 4 : MT];
    constexpr int MS = MT < 4 ? 4 : MT;
    const int col0 = (blockIdx.x * kPairThreads + threadIdx.x) * 2;
    const int m0 = blockIdx.y * MT;
    const int ca = min(col0, n - 1), cb = min(col0 + 1, n - 1);
    const int nbk = k / 32;
    const uint4* qa = reinterpret_cast<const uint4*>(quants) + static_cast<size_t>(ca) * (k / 16);
    const uint4* qb = reinterpret_cast<const uint4*>(quants) + static_cast<size_t>(cb) * (k / 16);

    float2 acc[MT];
#pragma unroll
    for (int r = 0; r < MT; ++r) acc[r] = make_float2(0.0f, 0.0f);

    for (int kc = 0; kc < k; kc += kPairKC) {
        const int kn = min(kPairKC, k - kc);
        __syncthreads();
        for (int e = threadIdx.x; e < kn * MS; e += kPairThreads) {
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
                    bs[r] = fadd2(bs[r], pair_products(xv.x, qq));
                    if (r + 1 < MT) bs[r + 1] = fadd2(bs[r + 1], pair_products(xv.y, qq));
                    if (r + 2 < MT) bs[r + 2] = fadd2(bs[r + 2], pair_products(xv.z, qq));
                    if (r + 3 < MT) bs[r + 3] = fadd2(bs[r + 3], pair_products(xv.w, qq));
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

// Stages the tile's activations x[m0 .. m0 + MT)[0 .. k) into xs as [k][MT] (x[m0 + r][kk] at
// kk*MT + r; rows past m as zeros): sixteen independent 16-byte loads per thread in flight when x
// is 16-byte aligned (item i = 4 consecutive k of row i % MT), else single floats.
template <int MT, int THREADS>
__device__ __forceinline__ void stage_x(float* xs, const float* __restrict__ x, int m, int m0, int k) {
    if ((reinterpret_cast<uintptr_t>(x) & 15) == 0) {
        const int items = MT * k / 4;
        for (int i0 = threadIdx.x; i0 < items; i0 += 16 * THREADS) {
            float4 v[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int i = i0 + u * THREADS;
                const int r = i % MT, k4 = i / MT;
                v[u] = (i < items && m0 + r < m)
                           ? __ldg(reinterpret_cast<const float4*>(x + static_cast<size_t>(m0 + r) * k) + k4)
                           : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            }
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int i = i0 + u * THREADS;
                if (i < items) {
                    const int r = i % MT, k4 = i / MT;
                    float* d = xs + (4 * k4) * MT + r;
                    d[0] = v[u].x;
                    d[MT] = v[u].y;
                    d[2 * MT] = v[u].z;
                    d[3 * MT] = v[u].w;
                }
            }
        }
    } else {
        const int total = MT * k;
        for (int e0 = threadIdx.x; e0 < total; e0 += 8 * THREADS) {
            float v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int e = e0 + u * THREADS;
                const int kk = e / MT, r = e % MT;
                v[u] = (e < total && m0 + r < m) ? __ldg(x + static_cast<size_t>(m0 + r) * k + kk) : 0.0f;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int e = e0 + u * THREADS;
                if (e < total) xs[e] = v[u];
            }
        }
    }
}

// 3 to 16 activation rows (a tile of MT of them per grid row): a warp owns a strip of 32 weight
// rows, one per lane, and runs every block of its row in order, so acc stays in a register and
// needs no hand-over.  The thread block stages the tile's activations once, [k][MT], and every
// read of them is a broadcast (all lanes at the same k).  Each lane streams its row's 32-byte
// blocks with D blocks in flight.  Four warps per thread block: the grid (n / 128 blocks
// per tile) is one wave with two or three thread blocks per SM.
constexpr int kStWarps = 4;
constexpr int kStDepth = 4;                    // blocks of codes in flight per lane (pairs)

template <int MT>
size_t st_smem(int k) { return static_cast<size_t>(k) * MT * 4; }
constexpr size_t kStSmemMax = 200 * 1024;

template <int MT, int W = kStWarps, int D = kStDepth>
__global__ void __launch_bounds__(W * 32)
block_q8_strip_kernel(const float* __restrict__ x, const uint32_t* __restrict__ quants,
                      const float* __restrict__ scales, float* __restrict__ y, int m, int k, int n) {
    extern __shared__ __align__(16) float smem_f[];          // [k][MT]: x[m0 + r][kk] at kk*MT + r
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nbk = k / 32;
    const int m0 = blockIdx.y * MT;
    const int row = (blockIdx.x * W + warp) * 32 + lane;
    const int rc = min(row, n - 1);                          // past-the-end rows: computed, not stored
    const uint4* qp = reinterpret_cast<const uint4*>(quants) + static_cast<size_t>(rc) * (k / 16);
    const float* sp = scales + static_cast<size_t>(rc) * nbk;

    // the first blocks' codes are requested before the wait for the preceding grids (weights are
    // not written by them); the activations are read after it
    uint4 w0[D], w1[D];
    float sc[D];
#pragma unroll
    for (int d = 0; d < D; ++d) {
        const int b = min(d, nbk - 1);
        w0[d] = __ldg(qp + 2 * b);
        w1[d] = __ldg(qp + 2 * b + 1);
        sc[d] = __ldg(sp + b);
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    stage_x<MT, W * 32>(smem_f, x, m, m0, k);
    __syncthreads();
    float acc[MT];
#pragma unroll
    for (int r = 0; r < MT; ++r) acc[r] = 0.0f;
    static_assert(D % 2 == 0, "blocks are summed in pairs");
    for (int b0 = 0; b0 < nbk; b0 += D) {
#pragma unroll
        for (int d = 0; d < D; d += 2) {             // slots d, d + 1 hold blocks b0 + d, b0 + d + 1
            const int b = b0 + d;
            if (b >= nbk) break;
            const bool two = b + 1 < nbk;
            uint32_t wq[2][8];
            float s[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                wq[h][0] = w0[d + h].x ^ 0x80808080u; wq[h][1] = w0[d + h].y ^ 0x80808080u;
                wq[h][2] = w0[d + h].z ^ 0x80808080u; wq[h][3] = w0[d + h].w ^ 0x80808080u;
                wq[h][4] = w1[d + h].x ^ 0x80808080u; wq[h][5] = w1[d + h].y ^ 0x80808080u;
                wq[h][6] = w1[d + h].z ^ 0x80808080u; wq[h][7] = w1[d + h].w ^ 0x80808080u;
                s[h] = sc[d + h];
                if (b + h + D < nbk) {                // refill the slot D blocks ahead
                    w0[d + h] = __ldg(qp + 2 * (b + h + D));
                    w1[d + h] = __ldg(qp + 2 * (b + h + D) + 1);
                    sc[d + h] = __ldg(sp + b + h + D);
                }
            }
            // the two blocks' sums are independent: their chains run side by side (a lone last
            // block sums block 0's activations in its second half, unused)
            const float* xb0 = smem_f + static_cast<size_t>(b) * 32 * MT;
            const float* xb1 = two ? xb0 + 32 * MT : smem_f;
            float bs0[MT], bs1[MT];
#pragma unroll
            for (int r = 0; r < MT; ++r) bs0[r] = bs1[r] = 0.0f;
#pragma unroll
            for (int t = 0; t < 32; ++t) {
                accumulate_rows<MT>(bs0, xb0 + t * MT, q_of(wq[0][t >> 2], t & 3));
                accumulate_rows<MT>(bs1, xb1 + t * MT, q_of(wq[1][t >> 2], t & 3));
            }
#pragma unroll
            for (int r = 0; r < MT; ++r) acc[r] = __fadd_rn(acc[r], __fmul_rn(s[0], bs0[r]));
            if (two) {
#pragma unroll
                for (int r = 0; r < MT; ++r) acc[r] = __fadd_rn(acc[r], __fmul_rn(s[1], bs1[r]));
            }
        }
    }
    // the next launch may start now (its prologue overlaps these stores); released only here so
    // that back-to-back launches do not pile up resident thread blocks that wait
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (row < n) {
#pragma unroll
        for (int r = 0; r < MT; ++r)
            if (m0 + r < m) y[static_cast<size_t>(m0 + r) * n + row] = acc[r];
    }
}

// The strip kernel with the codes brought in by the tensor-memory accelerator, persistent: one
// thread block per SM stages the tile's activations once, and takes an even share of the 32-row
// strips (ceil(n / 32) of them over the grid: every SM gets the same number to within one), its
// warps taking the block's strips in turn.  Each warp keeps a ring of S stages, one per 32-byte
// block, each the 32 x 32-byte tile of its strip's rows (1 KB, one tiled copy with the 32-byte
// swizzle, so each lane's two 16-byte reads of its row fall in distinct bank groups).  Lane 0
// refills a stage with the block S ahead as soon as the warp has read it, so S blocks of codes are
// in flight per warp without holding them in registers; the scales (4 bytes per row and block)
// are loaded by each lane S blocks ahead.  Every wait is bounded: a warp that gives up reports it,
// lets its copies still in flight land, and stops.
constexpr int kTmWarps = 11;                   // >= strips per SM for n up to 11 * 32 * SMs

template <int S, int W>
__host__ __device__ constexpr size_t tm_ring_bytes() { return static_cast<size_t>(W) * S * 1024; }
template <int S, int W>
__host__ __device__ constexpr size_t tm_bar_bytes() { return (static_cast<size_t>(W) * S * 8 + 15) / 16 * 16; }
template <int MT, int S, int W>
size_t tm_smem(int k) { return 1024 + tm_ring_bytes<S, W>() + tm_bar_bytes<S, W>() + static_cast<size_t>(k) * MT * 4; }
constexpr size_t kTmSmemOneBlock = 120 * 1024;   // requested at least: one thread block per SM

__device__ __forceinline__ uint4 lds128(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }

template <int MT, int S, int W = kTmWarps>
__global__ void __launch_bounds__(W * 32)
block_q8_tma_kernel(const __grid_constant__ CUtensorMap tm, const float* __restrict__ x,
                    const float* __restrict__ scales, float* __restrict__ y, int m, int k, int n) {
    static_assert(S % 2 == 0, "blocks are summed in pairs");
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint8_t* base = smem_align1024(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t* ring = base + static_cast<size_t>(warp) * S * 1024;
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + tm_ring_bytes<S, W>()) + warp * S;
    float* xs = reinterpret_cast<float*>(base + tm_ring_bytes<S, W>() + tm_bar_bytes<S, W>());
    const int nbk = k / 32;
    const int m0 = blockIdx.y * MT;
    const int strips = (n + 31) / 32;
    const int se = static_cast<int>(static_cast<long long>(blockIdx.x + 1) * strips / gridDim.x);
    const int sb = static_cast<int>(static_cast<long long>(blockIdx.x) * strips / gridDim.x);
    const bool busy = sb + warp < se;
    // ring of the warp's current strip: S blocks primed, phase counts per stage
    uint32_t ph[S];
#pragma unroll
    for (int d = 0; d < S; ++d) ph[d] = 0;
    auto prime = [&](int row0) {
        if (lane == 0) {
#pragma unroll
            for (int d = 0; d < S; ++d)
                if (d < nbk) {
                    mbar_arrive_expect_tx(&bars[d], 1024);
                    tma_load_2d(ring + d * 1024, &tm, 32 * d, row0, &bars[d]);
                }
        }
    };
    if (busy && lane == 0) {
        prefetch_tmap(&tm);
#pragma unroll
        for (int d = 0; d < S; ++d) mbar_init(&bars[d], 1);
        fence_barrier_init();
    }
    __syncwarp();
    // the first strip's first S blocks: before the wait for the preceding grids (weights)
    if (busy) prime((sb + warp) * 32);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    stage_x<MT, W * 32>(xs, x, m, m0, k);
    __syncthreads();
    for (int strip = sb + warp; strip < se; strip += W) {
        const int row0 = strip * 32;
        const int row = row0 + lane;
        const float* sp = scales + static_cast<size_t>(min(row, n - 1)) * nbk;   // past-the-end rows: not stored
        if (strip != sb + warp) prime(row0);      // the ring is empty: every copy of the last strip was used
        float sc[S];
#pragma unroll
        for (int d = 0; d < S; ++d) sc[d] = __ldg(sp + min(d, nbk - 1));
        float acc[MT];
#pragma unroll
        for (int r = 0; r < MT; ++r) acc[r] = 0.0f;
        for (int b0 = 0; b0 < nbk; b0 += S) {
#pragma unroll
            for (int d = 0; d < S; d += 2) {         // stages d, d + 1 hold blocks b0 + d, b0 + d + 1
                const int b = b0 + d;
                if (b >= nbk) break;
                const bool two = b + 1 < nbk;
                bool ok = __all_sync(0xffffffffu, mbar_wait(&bars[d], ph[d] & 1u));
                if (ok && two) ok = __all_sync(0xffffffffu, mbar_wait(&bars[d + 1], ph[d + 1] & 1u));
                if (!ok) {
                    if (lane == 0) {
                        report_error(kErrWaitTimeout);
                        // the copies still in flight: blocks [b, b + S) that exist, block c in stage
                        // c % S, each the next phase of its stage
#pragma unroll
                        for (int e = 0; e < S; ++e) {
                            const int c = b + ((e - d) + S) % S;
                            if (c < nbk && !mbar_wait(&bars[e], ph[e] & 1u)) report_error(kErrDrainTimeout);
                        }
                    }
                    return;                          // no block-wide barrier follows
                }
                ++ph[d];
                if (two) ++ph[d + 1];
                const uint4 a0 = lds128(ring + d * 1024 + swz32(lane, 0)), a1 = lds128(ring + d * 1024 + swz32(lane, 1));
                uint4 c0 = a0, c1 = a1;
                if (two) {
                    c0 = lds128(ring + (d + 1) * 1024 + swz32(lane, 0));
                    c1 = lds128(ring + (d + 1) * 1024 + swz32(lane, 1));
                }
                const float s0 = sc[d], s1 = sc[d + 1];
                if (b + S < nbk) sc[d] = __ldg(sp + b + S);
                if (b + 1 + S < nbk) sc[d + 1] = __ldg(sp + b + 1 + S);
                __syncwarp();                        // every lane has read the two stages
                if (lane == 0) {
                    fence_proxy_async_smem();
                    if (b + S < nbk) {
                        mbar_arrive_expect_tx(&bars[d], 1024);
                        tma_load_2d(ring + d * 1024, &tm, 32 * (b + S), row0, &bars[d]);
                    }
                    if (b + 1 + S < nbk) {
                        mbar_arrive_expect_tx(&bars[d + 1], 1024);
                        tma_load_2d(ring + (d + 1) * 1024, &tm, 32 * (b + 1 + S), row0, &bars[d + 1]);
                    }
                }
                const uint32_t wq[2][8] = {{a0.x ^ 0x80808080u, a0.y ^ 0x80808080u, a0.z ^ 0x80808080u, a0.w ^ 0x80808080u,
                                            a1.x ^ 0x80808080u, a1.y ^ 0x80808080u, a1.z ^ 0x80808080u, a1.w ^ 0x80808080u},
                                           {c0.x ^ 0x80808080u, c0.y ^ 0x80808080u, c0.z ^ 0x80808080u, c0.w ^ 0x80808080u,
                                            c1.x ^ 0x80808080u, c1.y ^ 0x80808080u, c1.z ^ 0x80808080u, c1.w ^ 0x80808080u}};
                // the two blocks' sums are independent: their chains run side by side (a lone last
                // block sums its own activations twice, the second copy unused)
                const float* xb0 = xs + static_cast<size_t>(b) * 32 * MT;
                const float* xb1 = two ? xb0 + 32 * MT : xb0;
                float bs0[MT], bs1[MT];
#pragma unroll
                for (int r = 0; r < MT; ++r) bs0[r] = bs1[r] = 0.0f;
#pragma unroll
                for (int t = 0; t < 32; ++t) {
                    accumulate_rows<MT>(bs0, xb0 + t * MT, q_of(wq[0][t >> 2], t & 3));
                    accumulate_rows<MT>(bs1, xb1 + t * MT, q_of(wq[1][t >> 2], t & 3));
                }
#pragma unroll
                for (int r = 0; r < MT; ++r) acc[r] = __fadd_rn(acc[r], __fmul_rn(s0, bs0[r]));
                if (two) {
#pragma unroll
                    for (int r = 0; r < MT; ++r) acc[r] = __fadd_rn(acc[r], __fmul_rn(s1, bs1[r]));
                }
            }
        }
        if (strip + W >= se) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");   // last strip
        if (row < n) {
#pragma unroll
            for (int r = 0; r < MT; ++r)
                if (m0 + r < m) y[static_cast<size_t>(m0 + r) * n + row] = acc[r];
        }
    }
}

// The tensor-memory-accelerator strip kernel when its shared memory fits and the driver encodes
// the codes' tensor map ([n] rows of k bytes, 32 x 32-byte boxes, 32-byte swizzle); returns
// cudaErrorNotSupported otherwise, so the caller can take the register-streaming kernel.  One
// thread block per SM and tile of MT activation rows.
template <int MT, int S, int W = kTmWarps>
cudaError_t launch_tma(const float* x, const uint32_t* q, const float* s, float* y, int m, int k, int n,
                       cudaStream_t st) {
    const size_t need = tm_smem<MT, S, W>(k);
    if (need > kStSmemMax) return cudaErrorNotSupported;
    const size_t smem = need < kTmSmemOneBlock ? kTmSmemOneBlock : need;
    CUtensorMap tm;
    if (!make_tmap_2d_swizzle(&tm, q, CU_TENSOR_MAP_DATA_TYPE_UINT8, static_cast<uint64_t>(k), static_cast<uint64_t>(n),
                              static_cast<uint64_t>(k), 32, 32, CU_TENSOR_MAP_SWIZZLE_32B))
        return cudaErrorNotSupported;
    static int configured_dev = -1, sms = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_dev != dev) {
        e = cudaFuncSetAttribute(block_q8_tma_kernel<MT, S, W>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kStSmemMax));
        if (e != cudaSuccess) return e;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        configured_dev = dev;
    }
    const int strips = (n + 31) / 32;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(strips < sms ? strips : sms, (m + MT - 1) / MT);
    cfg.blockDim = dim3(W * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, block_q8_tma_kernel<MT, S, W>, tm, x, s, y, m, k, n);
}

template <int MT>
cudaError_t launch_strip(const float* x, const uint32_t* q, const float* s, float* y, int m, int k, int n,
                         cudaStream_t st) {
    static int configured_dev = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_dev != dev) {
        e = cudaFuncSetAttribute(block_q8_strip_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kStSmemMax));
        if (e != cudaSuccess) return e;
        configured_dev = dev;
    }
    // a programmatic dependent of the previous launch on the stream (see the kernel)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((n + kStWarps * 32 - 1) / (kStWarps * 32), (m + MT - 1) / MT);
    cfg.blockDim = dim3(kStWarps * 32);
    cfg.dynamicSmemBytes = st_smem<MT>(k);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, block_q8_strip_kernel<MT>, x, q, s, y, m, k, n);
}

template <int MT>
cudaError_t launch_mt(const float* x, const uint32_t* q, const float* s, float* y, int m, int k, int n,
                      cudaStream_t st) {
    if constexpr (MT >= 8) {
        const dim3 grid((n + 2 * kPairThreads - 1) / (2 * kPairThreads), (m + MT - 1) / MT);
        block_q8_pair_kernel<MT><<<grid, kPairThreads, 0, st>>>(x, q, s, y, m, k, n);
    } else {
        static int configured_dev = -1;
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (configured_dev != dev) {
            e = cudaFuncSetAttribute(block_q8_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(bq8_smem<MT>(1 << 30)));
            if (e != cudaSuccess) return e;
            configured_dev = dev;
        }
        const dim3 grid((n + kColsPerCta - 1) / kColsPerCta, (m + MT - 1) / MT);
        block_q8_kernel<MT><<<grid, warps_of<MT>() * 32, bq8_smem<MT>(k), st>>>(x, q, s, y, m, k, n);
    }
    return cudaGetLastError();
}

}  // namespace

GQ_ERROR_ACCESSOR(block_q8)

cudaError_t launch_block_q8(const float* x, const uint32_t* quants, const float* scales, float* y, int m, int k,
                            int n, cudaStream_t s) {
    if (m == 2) {
        const cudaError_t e = launch_tma<2, 4>(x, quants, scales, y, m, k, n, s);
        if (e != cudaErrorNotSupported) return e;
    }
    if (m <= 2) {
        // x rows 16-byte aligned for the activations' vector loads (k % 32 == 0 and x 16-aligned)
        if ((reinterpret_cast<uintptr_t>(x) & 15) == 0) {
            cudaLaunchConfig_t cfg = {};
            cfg.blockDim = dim3(kRwWarps * 32);
            cfg.stream = s;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[0].val.programmaticStreamSerializationAllowed = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            if (m == 1) {
                constexpr int rows = kRwWarps * rw_rows<1>();
                cfg.gridDim = dim3((n + rows - 1) / rows);
                return cudaLaunchKernelEx(&cfg, block_q8_rowwarp_kernel<1>, x, quants, scales, y, m, k, n);
            }
            constexpr int rows = kRwWarps * rw_rows<2>();
            cfg.gridDim = dim3((n + rows - 1) / rows);
            return cudaLaunchKernelEx(&cfg, block_q8_rowwarp_kernel<2>, x, quants, scales, y, m, k, n);
        }
        return m <= 1 ? launch_mt<1>(x, quants, scales, y, m, k, n, s) : launch_mt<2>(x, quants, scales, y, m, k, n, s);
    }
    // 3 or more rows: the strip kernels while the staged activations fit in shared memory (the
    // TMA-fed one for tiles of 4 and 16 rows, where it measured faster; the register-streaming one
    // for 8 and whenever the tensor map cannot be encoded), else the pass kernels.
    if (m <= 4) {
        const cudaError_t e = launch_tma<4, 4>(x, quants, scales, y, m, k, n, s);
        if (e != cudaErrorNotSupported) return e;
        return st_smem<4>(k) <= kStSmemMax ? launch_strip<4>(x, quants, scales, y, m, k, n, s)
                                           : launch_mt<4>(x, quants, scales, y, m, k, n, s);
    }
    if (m <= 8) return st_smem<8>(k) <= kStSmemMax ? launch_strip<8>(x, quants, scales, y, m, k, n, s)
                                                  : launch_mt<8>(x, quants, scales, y, m, k, n, s);
    const cudaError_t e = launch_tma<16, 2>(x, quants, scales, y, m, k, n, s);
    if (e != cudaErrorNotSupported) return e;
    return st_smem<16>(k) <= kStSmemMax ? launch_strip<16>(x, quants, scales, y, m, k, n, s)
                                        : launch_mt<16>(x, quants, scales, y, m, k, n, s);
}

}  // namespace gq
