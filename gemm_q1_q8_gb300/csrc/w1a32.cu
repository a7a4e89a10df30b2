// Bonsai 1-bit weights times f32 activations on sm_103a (BonsaiのWebGPUカーネルを読み解く, the
// decode/prefill figure).  The weights are the Bonsai format -- one u32 of 32 sign bits (bit 1 ->
// +1.0, bit 0 -> -1.0) and one f32 scale per 32 weights -- and
//   y[m, n] = sum_b ws[n, b] * sum_t s(n, 32 b + t) * x[m, 32 b + t].
// The page gives two formulations and fixes the order of the float operations in neither, so the
// results are checked against the exact value within an error bound of the kernel's own order.
//
// FMA path (the page's decode kernel, llama-decode-q1-proj.wgsl): signs expanded to +-1 and
// summed, one activation read serving four rows.  A warp covers four weight rows, each lane the
// blocks lane, lane + 32, ... of those rows.  The activations sit in shared memory transposed
// ([t][block], stride odd) so the lanes' reads of consecutive blocks are conflict-free; the sign is
// applied by flipping the float's sign bit (a row's word shifted so bit t lands on bit 31).  Each
// lane sums a block's 32 signed activations in order, then acc = fma(scale, d, acc) over its blocks,
// and a butterfly over the warp's lanes adds the lanes.
//
// LUT4 path (the page's prefill kernel, binary-lut4-matmul.wgsl): per token and four activations
// a table of the 16 signed sums +-x0 +-x1 +-x2 +-x3, indexed by the weight nibble (bit k of the
// nibble -> the sign of x_k), built once in shared memory and read by every row of the thread
// block.  The lanes of a warp are 32 rows reading the same table, so a lookup touches at most 16
// distinct words -- no bank conflicts.  A table entry is (+-x0 +-x1) + (+-x2 +-x3); a block sum is
// the eight lookups added in nibble order; acc = fma(scale, block_sum, acc) in block order.
//   * decode (M <= 4): a thread block covers 32 rows, its eight warps split the blocks of K and
//     add their partial results in a fixed tree; the entries hold the M tokens side by side.
//   * prefill (M > 4): a thread block covers 256 rows x 4*MQ tokens; the entries hold four
//     tokens, and only eight are stored per group -- s(15 - i) = -s(i), so a nibble with its top
//     bit set reads entry (i ^ 15) and multiplies by -1 (exact), which halves the shared-memory
//     bytes per lookup.
#include <cooperative_groups.h>

#include "gq_internal.cuh"

namespace cg = cooperative_groups;

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


// ------------------------------------------------------------------------------------ LUT4 path

template <int T> struct FVec;                     // T tokens side by side in one table entry
template <> struct FVec<1> { float v[1]; };
template <> struct alignas(8) FVec<2> { float v[2]; };
template <> struct alignas(16) FVec<4> { float v[4]; };

template <int T>
__device__ __forceinline__ FVec<T> lds_vec(const FVec<T>* p) {
    FVec<T> r;
    if constexpr (T == 1) {
        r.v[0] = *reinterpret_cast<const float*>(p);
    } else if constexpr (T == 2) {
        const float2 a = *reinterpret_cast<const float2*>(p);
        r.v[0] = a.x; r.v[1] = a.y;
    } else {
        const float4 a = *reinterpret_cast<const float4*>(p);
        r.v[0] = a.x; r.v[1] = a.y; r.v[2] = a.z; r.v[3] = a.w;
    }
    return r;
}
template <int T>
__device__ __forceinline__ void sts_vec(FVec<T>* p, const float (&v)[T]) {
    if constexpr (T == 1) *reinterpret_cast<float*>(p) = v[0];
    else if constexpr (T == 2) *reinterpret_cast<float2*>(p) = make_float2(v[0], v[1]);
    else *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
}

// The four activations x[32 b + 4 g .. + 3] of one token.
__device__ __forceinline__ float4 ldg_x4(const float* x, size_t m, int K, int b, int g) {
    return __ldg(reinterpret_cast<const float4*>(x + m * static_cast<size_t>(K) + static_cast<size_t>(b) * 32 + 4 * g));
}

// A group's table is padded by one entry, so the builders' stores (one table per lane) hit
// distinct banks; the lookups of one group still read 16 consecutive entries.
constexpr int kDecTab = 17;

__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
constexpr int kDecRows = 128;                     // rows per thread block: four warps of 32
constexpr int kDecStage = 32;                     // blocks per stage: one 128-byte row of words
constexpr int kDecMaxSlices = 8;                  // K slices = thread blocks of one cluster

template <int T>
struct DecLayout {
    static constexpr uint32_t sig = 0;                                   // [128 rows][32 words], 128B swizzle
    static constexpr uint32_t sc = sig + kDecRows * kDecStage * 4;       // [128 rows][32 scales], same
    static constexpr uint32_t part = sig;                                // [2 halves][128 rows], after the last stage
    static constexpr uint32_t lut = sc + kDecRows * kDecStage * 4;       // [32 blocks][8 groups][kDecTab]
    static constexpr uint32_t bar = lut + kDecStage * 8 * kDecTab * sizeof(FVec<T>);   // one per 32-row group
    static constexpr uint32_t flag = bar + 4 * 8;
    static constexpr uint32_t cl = flag + 16;                            // [slice][128 rows], filled in rank 0
    static constexpr uint32_t bytes(int slices) {
        return cl + static_cast<uint32_t>(slices) * kDecRows * sizeof(FVec<T>);
    }
};

// One warp's share of a stage: blocks 16*H .. 16*H + 15 of the stage (fewer in a short stage),
// for the warp's 32 rows.  H is a template argument so every table address is a constant offset.
template <int T, int H>
__device__ __forceinline__ void dec_consume(const uint8_t* base, const FVec<T>* lut, int row, int nbs,
                                            float (&acc)[T]) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int j0 = 16 * H + 4 * c;
        if (j0 >= nbs) break;
        const uint32_t off = swz128(row, 4 * H + c);
        const uint4 wq = *reinterpret_cast<const uint4*>(base + DecLayout<T>::sig + off);
        const float4 sq = *reinterpret_cast<const float4*>(base + DecLayout<T>::sc + off);
        const uint32_t wv[4] = {wq.x, wq.y, wq.z, wq.w};
        const float sv[4] = {sq.x, sq.y, sq.z, sq.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if (j0 + k < nbs) {
                const uint32_t w = wv[k];
                const FVec<T>* tb = lut + (j0 + k) * 8 * kDecTab;
                FVec<T> S = lds_vec<T>(tb + (w & 15u));
#pragma unroll
                for (int g = 1; g < 8; ++g) {
                    const FVec<T> L = lds_vec<T>(tb + g * kDecTab + ((w >> (4 * g)) & 15u));
#pragma unroll
                    for (int u = 0; u < T; ++u) S.v[u] = __fadd_rn(S.v[u], L.v[u]);
                }
#pragma unroll
                for (int u = 0; u < T; ++u) acc[u] = __fmaf_rn(sv[k], S.v[u], acc[u]);
            }
        }
    }
}

// Decode, M <= T tokens (T = 1, 2, 4).  A cluster of `gridDim.y` thread blocks covers 128 rows;
// block r of it takes the K slice [r*ks, (r+1)*ks) (ks a multiple of 4 blocks), staged 32 blocks
// at a time: per 32-row group one TMA copy of the rows' sign words and one of their scales, on the
// group's own barrier, while the threads build the slice's tables from x; the warps of a group
// start on their rows as soon as those have landed.  Warps 0-3 take blocks 0-15 of a stage, warps 4-7 blocks
// 16-31, for rows 32*(warp & 3) + lane.  The two halves are added, every block stores its sums
// into block 0's shared memory (distributed shared memory), and block 0 adds the slices in slice
// order and stores y.
template <int T>
__global__ void __launch_bounds__(256)
lut4_decode_kernel(const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmW,
                   const float* __restrict__ x, float* __restrict__ y, int N, int K, int M, int ks) {
    using L = DecLayout<T>;
    extern __shared__ __align__(1024) uint8_t dsm[];
    uint8_t* base = smem_align1024(dsm);
    FVec<T>* lut = reinterpret_cast<FVec<T>*>(base + L::lut);
    FVec<T>* part = reinterpret_cast<FVec<T>*>(base + L::part);
    FVec<T>* cl = reinterpret_cast<FVec<T>*>(base + L::cl);
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + L::bar);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base + L::flag);
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());
    const int nsl = static_cast<int>(cluster.num_blocks());
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = warp >> 2, row = (warp & 3) * 32 + lane;
    const int row0 = blockIdx.x * kDecRows;
    const int nbk = K / 32;
    const int s_lo = rank * ks, s_hi = min(s_lo + ks, nbk);
    if (threadIdx.x == 0) {
        prefetch_tmap(&tmS);
        prefetch_tmap(&tmW);
        for (int g = 0; g < 4; ++g) mbar_init(&bars[g], 1);
        fence_barrier_init();
        *abort_flag = 0;
    }
    __syncthreads();
    cluster_arrive_relaxed();                     // waited for before the first remote store
    float acc[T];
#pragma unroll
    for (int u = 0; u < T; ++u) acc[u] = 0.0f;
    uint32_t phase = 0, issued_parity = 0;
    bool issued = false;
    for (int b0 = s_lo; b0 < s_hi; b0 += kDecStage) {
        const int nbs = min(kDecStage, s_hi - b0);
        if (threadIdx.x == 0 && !*abort_flag) {
            issued = true;
            issued_parity = phase;
            for (int g = 0; g < 4; ++g) {
                mbar_arrive_expect_tx(&bars[g], 2u * 32 * kDecStage * 4);
                tma_load_2d(base + L::sig + g * 32 * 128, &tmS, b0, row0 + 32 * g, &bars[g]);
                tma_load_2d(base + L::sc + g * 32 * 128, &tmW, b0, row0 + 32 * g, &bars[g]);
            }
        }
        {   // tables of this stage: one (block, group) per thread
            const int j = threadIdx.x >> 3, g = threadIdx.x & 7;
            if (j < nbs) {
                float e[16][T];
#pragma unroll
                for (int u = 0; u < T; ++u) {
                    const float4 a = ldg_x4(x, min(u, M - 1), K, b0 + j, g);
                    // p(i0 i1) = +-x0 +-x1, q(i2 i3) = +-x2 +-x3 (bit set -> +)
                    const float p0 = -(a.x + a.y), p1 = a.x - a.y;
                    const float q0 = -(a.z + a.w), q1 = a.z - a.w;
                    const float p[4] = {p0, p1, -p1, -p0};
                    const float qq[4] = {q0, q1, -q1, -q0};
#pragma unroll
                    for (int i = 0; i < 16; ++i) e[i][u] = __fadd_rn(p[i & 3], qq[i >> 2]);
                }
                FVec<T>* dst = lut + threadIdx.x * kDecTab;
#pragma unroll
                for (int i = 0; i < 16; ++i) sts_vec<T>(dst + i, e[i]);
            }
        }
        __syncthreads();
        if (!*abort_flag) {
            if (!mbar_wait(&bars[warp & 3], phase)) {
                report_error(kErrWaitTimeout);
                *abort_flag = 1;
            }
        }
        if (!*abort_flag) {
            if (h == 0) dec_consume<T, 0>(base, lut, row, nbs, acc);
            else dec_consume<T, 1>(base, lut, row, nbs, acc);
        }
        phase ^= 1u;
        __syncthreads();                          // buffers and tables free for the next stage
    }
    if (*abort_flag && threadIdx.x == 0 && issued) {
        // the last copy may still be landing: let it finish (bounded) before the block can exit
        for (int g = 0; g < 4; ++g)
            if (!mbar_wait(&bars[g], issued_parity)) report_error(kErrDrainTimeout);
    }
    __syncthreads();
    sts_vec<T>(part + h * kDecRows + row, acc);
    __syncthreads();
    cluster_wait();                               // every block of the cluster has started
    if (h == 0) {
        const FVec<T> a = lds_vec<T>(part + row), b = lds_vec<T>(part + kDecRows + row);
        float v[T];
#pragma unroll
        for (int u = 0; u < T; ++u) v[u] = __fadd_rn(a.v[u], b.v[u]);
        sts_vec<T>(cluster.map_shared_rank(cl, 0) + rank * kDecRows + row, v);
    }
    cluster_arrive_release();
    if (rank == 0) {
        cluster_wait_acquire();                   // all slices' sums are in this block
        if (h == 0 && row0 + row < N) {
            FVec<T> v = lds_vec<T>(cl + row);
            for (int r = 1; r < nsl; ++r) {
                const FVec<T> o = lds_vec<T>(cl + r * kDecRows + row);
#pragma unroll
                for (int u = 0; u < T; ++u) v.v[u] = __fadd_rn(v.v[u], o.v[u]);
            }
#pragma unroll
            for (int u = 0; u < T; ++u)
                if (u < M) y[static_cast<size_t>(u) * N + row0 + row] = v.v[u];
        }
    }
    // the other blocks leave: nothing reads their shared memory
}

// Decode of one token, persistent: one thread block per SM takes 32-row tiles in turn.  A tile's
// sign words and scales come by TMA (four 128-byte-wide boxes of 32 rows each, 128B swizzle) into a
// three-stage ring, two tiles ahead of the one being summed.  The sixteen warps split a tile's
// blocks (warp w the blocks w*nb/16 ...), each lane one row, and each warp builds the tables of its
// own blocks only (the activation is the same for every row), so no warp waits for another before
// its first tile.  The warps' partial sums are added in a fixed tree.  When a block has at most
// three tiles (the usual case), each tile keeps its own stage and partial-sum slot and the block
// meets at a barrier only once, at the end.
// Launched as a programmatic dependent: the first two tiles' copies are requested before the wait
// for the preceding grids, the activations (tables) read and the outputs written after it.  The
// third tile is requested once warp 0 has built its tables, so that the activation reads after the
// wait do not queue behind a whole call's weight stream (5.23 -> 4.97 us at 14,336 x 4,096).
constexpr int kPdWarps = 16;
constexpr int kPdStages = 3;
constexpr int kPdMaxBlocks = 160;                 // K <= 5120: the tables fit beside the ring
constexpr int kPdBoxWords = 32;                   // words per TMA box row (128 bytes)

struct PdLayout {
    uint32_t ring, lut, part, bar, bytes;
};
__host__ __device__ inline PdLayout pd_layout(int nbk) {
    PdLayout L{};
    const uint32_t boxes = static_cast<uint32_t>((nbk + kPdBoxWords - 1) / kPdBoxWords);
    const uint32_t stage = 2u * boxes * 32u * 128u;                      // signs then scales
    L.ring = 0;
    L.lut = kPdStages * stage;
    L.part = L.lut + static_cast<uint32_t>(nbk) * 8u * kDecTab * 4u;
    L.part = (L.part + 15u) & ~15u;
    L.bar = L.part + kPdStages * kPdWarps * 32u * 4u;                   // one partial-sum slot per stage
    L.bytes = L.bar + kPdStages * 8u;
    return L;
}

// The warps' partial sums of one 32-row tile, added in a fixed tree, then stored.
__device__ __forceinline__ void pd_reduce_store(const float* part, int t, int lane, float* y, int N) {
    float v[kPdWarps];
#pragma unroll
    for (int w2 = 0; w2 < kPdWarps; ++w2) v[w2] = part[w2 * 32 + lane];
#pragma unroll
    for (int h = kPdWarps / 2; h >= 1; h >>= 1)
#pragma unroll
        for (int w2 = 0; w2 < h; ++w2) v[w2] = __fadd_rn(v[w2], v[w2 + h]);
    const int n = t * 32 + lane;
    if (n < N) y[n] = v[0];
}

__global__ void __launch_bounds__(kPdWarps * 32, 1)
lut4_decode_persistent_kernel(const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmW,
                              const float* __restrict__ x, float* __restrict__ y, int N, int K) {
    extern __shared__ __align__(1024) uint8_t psm1[];
    uint8_t* base = smem_align1024(psm1);
    const int nbk = K / 32;
    const PdLayout L = pd_layout(nbk);
    const int boxes = (nbk + kPdBoxWords - 1) / kPdBoxWords;
    const uint32_t half = static_cast<uint32_t>(boxes) * 32u * 128u;    // bytes of one tensor in a stage
    float* lut = reinterpret_cast<float*>(base + L.lut);                 // [block][group][kDecTab]
    float* part = reinterpret_cast<float*>(base + L.part);               // [stage][warp][lane]
    uint64_t* full = reinterpret_cast<uint64_t*>(base + L.bar);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tiles = (N + 31) / 32;
    const int my_tiles = (tiles - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                         static_cast<int>(gridDim.x);
    // every tile of this block has its own stage and partial-sum slot: no block-wide barrier until
    // the end (the usual case: 14,336 rows are 448 tiles, at most three per block)
    const bool oneshot = my_tiles <= kPdStages;

    auto issue = [&](int t, int s) {              // thread 0: tile t into stage s
        mbar_arrive_expect_tx(&full[s], 2u * half);
        for (int bx = 0; bx < boxes; ++bx) {
            tma_load_2d(base + L.ring + s * 2u * half + bx * 4096u, &tmS, bx * kPdBoxWords, t * 32, &full[s]);
            tma_load_2d(base + L.ring + s * 2u * half + half + bx * 4096u, &tmW, bx * kPdBoxWords, t * 32, &full[s]);
        }
    };
    int issued = 0;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (threadIdx.x == 0) {
        prefetch_tmap(&tmS);
        prefetch_tmap(&tmW);
        for (int s = 0; s < kPdStages; ++s) mbar_init(&full[s], 1);
        fence_barrier_init();
        for (int j = 0; j < 2; ++j) {
            const int t = blockIdx.x + j * gridDim.x;
            if (t < tiles) {
                issue(t, j);
                ++issued;
            }
        }
    }
    __syncthreads();                                         // the barriers are initialised
    asm volatile("griddepcontrol.wait;" ::: "memory");       // the preceding grids are done
    // whole 16-byte chunks (four blocks) per warp: nbk is a multiple of 4 (K % 128 == 0)
    const int per = ((nbk + kPdWarps - 1) / kPdWarps + 3) & ~3;
    const int jlo = warp * per, cnt = max(0, min(per, nbk - jlo));
    // each warp builds the tables of its own blocks (no other warp reads them): one (block, group) per item
    for (int it = lane; it < cnt * 8; it += 32) {
        const int j = jlo + (it >> 3), g = it & 7;
        const float4 a = ldg_x4(x, 0, K, j, g);
        const float p0 = -(a.x + a.y), p1 = a.x - a.y;
        const float q0 = -(a.z + a.w), q1 = a.z - a.w;
        const float p[4] = {p0, p1, -p1, -p0};
        const float qq[4] = {q0, q1, -q1, -q0};
        float* dst = lut + static_cast<size_t>(j * 8 + g) * kDecTab;
#pragma unroll
        for (int i = 0; i < 16; ++i) dst[i] = __fadd_rn(p[i & 3], qq[i >> 2]);
    }
    __syncwarp();
    if (threadIdx.x == 0) {                       // the third tile, after this warp's activation reads
        for (int j = 2; j < kPdStages; ++j) {
            const int t = blockIdx.x + j * gridDim.x;
            if (t < tiles) {
                issue(t, j);
                ++issued;
            }
        }
    }

    int i = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++i) {
        const int s = i % kPdStages;
        bool ok;
        if (oneshot) {
            ok = __all_sync(0xffffffffu, mbar_wait(&full[s], static_cast<uint32_t>(i / kPdStages) & 1u));
            if (!ok && lane == 0) report_error(kErrWaitTimeout);
        } else {
            ok = mbar_wait(&full[s], static_cast<uint32_t>(i / kPdStages) & 1u);
            if (__syncthreads_or(!ok)) {
                if (threadIdx.x == 0) report_error(kErrWaitTimeout);
                break;
            }
        }
        const uint8_t* sig = base + L.ring + s * 2u * half;
        const uint8_t* scl = sig + half;
        float acc = 0.0f;
        for (int j4 = jlo; ok && j4 < jlo + cnt; j4 += 4) {
            // four blocks' words and scales: one 16-byte chunk of the lane's row in each (swizzled)
            const uint32_t off = static_cast<uint32_t>(j4 / kPdBoxWords) * 4096u + static_cast<uint32_t>(lane) * 128u +
                                 ((static_cast<uint32_t>((j4 % kPdBoxWords) >> 2) ^ static_cast<uint32_t>(lane & 7)) << 4);
            const uint4 w4 = *reinterpret_cast<const uint4*>(sig + off);
            const float4 s4 = *reinterpret_cast<const float4*>(scl + off);
            const uint32_t wv[4] = {w4.x, w4.y, w4.z, w4.w};
            const float sv[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
                const uint32_t w = wv[k4];
                const float* tb = lut + static_cast<size_t>(j4 + k4) * 8 * kDecTab;
                float S = tb[w & 15u];
#pragma unroll
                for (int g = 1; g < 8; ++g) S = __fadd_rn(S, tb[g * kDecTab + ((w >> (4 * g)) & 15u)]);
                acc = __fmaf_rn(sv[k4], S, acc);
            }
        }
        if (oneshot) {
            part[(s * kPdWarps + warp) * 32 + lane] = acc;
            continue;
        }
        part[warp * 32 + lane] = acc;
        __syncthreads();
        if (warp == 0) pd_reduce_store(part, t, lane, y, N);
        __syncthreads();                          // stage s and the partial sums are free
        if (threadIdx.x == 0 && t + kPdStages * static_cast<int>(gridDim.x) < tiles) {
            issue(t + kPdStages * gridDim.x, s);
            ++issued;
        }
    }
    if (oneshot) {
        __syncthreads();
        if (warp < my_tiles)                      // warp w adds tile w's partial sums
            pd_reduce_store(part + warp * kPdWarps * 32, static_cast<int>(blockIdx.x) + warp * static_cast<int>(gridDim.x),
                            lane, y, N);
    }
    if (threadIdx.x == 0) {
        // after an early exit, copies still in flight land before shared memory is released
        // (in the one-shot case every stage was used once, and a completed phase is seen at once)
        for (int j = oneshot ? 0 : i; j < issued; ++j)
            if (!mbar_wait(&full[j % kPdStages], static_cast<uint32_t>(j / kPdStages) & 1u))
                report_error(kErrDrainTimeout);
    }
}

constexpr int kPreWarps = 8;
constexpr int kPreRows = kPreWarps * 32;          // one row per lane
constexpr int kPreStage = 4;                      // blocks per stage
constexpr int kPreTab = 9;                        // eight entries per group, padded by one (as above)

template <int MQ>
constexpr size_t pre_smem_bytes() { return static_cast<size_t>(MQ) * kPreStage * 8 * kPreTab * sizeof(float4); }

// Prefill: a thread block covers 256 rows x 4*MQ tokens.  Folded tables: entry i < 8 of a group
// holds s(i) = (+-x0 +-x1) + (+-x2 - x3) for four tokens.
template <int MQ>
__global__ void __launch_bounds__(kPreRows, 2)
lut4_prefill_kernel(const uint32_t* __restrict__ signs, const float* __restrict__ ws, const float* __restrict__ x,
                    float* __restrict__ y, int N, int K, int M) {
    extern __shared__ __align__(16) uint8_t psm[];
    float4* lut = reinterpret_cast<float4*>(psm);          // [quad][block][group][kPreTab]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = blockIdx.x * kPreRows + warp * 32 + lane;
    const int nc = min(n, N - 1);
    const int m0 = blockIdx.y * 4 * MQ;
    const int nbk = K / 32;
    const uint32_t* srow = signs + static_cast<size_t>(nc) * nbk;
    const float* wrow = ws + static_cast<size_t>(nc) * nbk;
    const bool vec = (((reinterpret_cast<uintptr_t>(srow) | reinterpret_cast<uintptr_t>(wrow)) & 15) == 0);

    // table builder item of this thread: (quad, block, group); MQ * 32 items
    const int iq = threadIdx.x >> 5, ij = (threadIdx.x >> 3) & 3, ig = threadIdx.x & 7;
    const bool builder = iq < MQ;
    int tok[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) tok[u] = min(m0 + 4 * iq + u, M - 1);

    auto load_w = [&](int b0, uint32_t (&wd)[kPreStage], float (&sc)[kPreStage]) {
        if (vec && b0 + kPreStage <= nbk) {
            const uint4 a = __ldg(reinterpret_cast<const uint4*>(srow + b0));
            const float4 c = __ldg(reinterpret_cast<const float4*>(wrow + b0));
            wd[0] = a.x; wd[1] = a.y; wd[2] = a.z; wd[3] = a.w;
            sc[0] = c.x; sc[1] = c.y; sc[2] = c.z; sc[3] = c.w;
        } else {
#pragma unroll
            for (int j = 0; j < kPreStage; ++j) {
                wd[j] = (b0 + j < nbk) ? __ldg(srow + b0 + j) : 0u;
                sc[j] = (b0 + j < nbk) ? __ldg(wrow + b0 + j) : 0.0f;
            }
        }
    };
    auto load_x = [&](int b0, float4 (&xa)[4]) {
        if (builder && b0 + ij < nbk) {
#pragma unroll
            for (int u = 0; u < 4; ++u) xa[u] = ldg_x4(x, tok[u], K, b0 + ij, ig);
        }
    };

    float4 acc[MQ];
#pragma unroll
    for (int q = 0; q < MQ; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
    uint32_t wn[kPreStage];
    float sn[kPreStage];
    float4 xn[4];
    load_w(0, wn, sn);
    load_x(0, xn);

    for (int b0 = 0; b0 < nbk; b0 += kPreStage) {
        uint32_t wd[kPreStage];
        float sc[kPreStage];
        float4 xa[4];
#pragma unroll
        for (int j = 0; j < kPreStage; ++j) { wd[j] = wn[j]; sc[j] = sn[j]; }
#pragma unroll
        for (int u = 0; u < 4; ++u) xa[u] = xn[u];
        if (b0 + kPreStage < nbk) {
            load_w(b0 + kPreStage, wn, sn);
            load_x(b0 + kPreStage, xn);
        }
        __syncthreads();                          // the previous stage's tables are no longer read
        if (builder && b0 + ij < nbk) {
            float e[8][4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float4 a = xa[u];
                const float p0 = -(a.x + a.y), p1 = a.x - a.y;
                const float r0 = -(a.z + a.w), r1 = a.z - a.w;     // x3 enters with a minus sign
                const float p[4] = {p0, p1, -p1, -p0};
#pragma unroll
                for (int i = 0; i < 8; ++i) e[i][u] = __fadd_rn(p[i & 3], (i & 4) ? r1 : r0);
            }
            float4* dst = lut + static_cast<size_t>(threadIdx.x) * kPreTab;
#pragma unroll
            for (int i = 0; i < 8; ++i) dst[i] = make_float4(e[i][0], e[i][1], e[i][2], e[i][3]);
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < kPreStage; ++j) {
            if (b0 + j < nbk) {
                const uint32_t w = wd[j];
                // nibble g -> folded index (low three bits, flipped when the top bit is set)
                const uint32_t h = (w >> 3) & 0x11111111u;
                const uint32_t f = (w ^ (h * 7u)) & 0x77777777u;
                int off[8];
                float sg[8];
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                    off[g] = g * kPreTab + static_cast<int>((f >> (4 * g)) & 7u);
                    sg[g] = __uint_as_float(0x3F800000u | ((w << (28 - 4 * g)) & 0x80000000u));
                }
                const float2 s2 = make_float2(sc[j], sc[j]);
#pragma unroll
                for (int q = 0; q < MQ; ++q) {
                    const float4* tb = lut + static_cast<size_t>(q * kPreStage + j) * 8 * kPreTab;
                    float4 L = tb[off[0]];
                    float2 Slo = fmul2(make_float2(sg[0], sg[0]), make_float2(L.x, L.y));
                    float2 Shi = fmul2(make_float2(sg[0], sg[0]), make_float2(L.z, L.w));
#pragma unroll
                    for (int g = 1; g < 8; ++g) {
                        L = tb[off[g]];
                        const float2 s = make_float2(sg[g], sg[g]);
                        Slo = ffma2(s, make_float2(L.x, L.y), Slo);
                        Shi = ffma2(s, make_float2(L.z, L.w), Shi);
                    }
                    const float2 alo = ffma2(s2, Slo, make_float2(acc[q].x, acc[q].y));
                    const float2 ahi = ffma2(s2, Shi, make_float2(acc[q].z, acc[q].w));
                    acc[q] = make_float4(alo.x, alo.y, ahi.x, ahi.y);
                }
            }
        }
    }
    if (n < N) {
#pragma unroll
        for (int q = 0; q < MQ; ++q) {
            const float a[4] = {acc[q].x, acc[q].y, acc[q].z, acc[q].w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int m = m0 + 4 * q + u;
                if (m < M) y[static_cast<size_t>(m) * N + n] = a[u];
            }
        }
    }
}

template <typename Kern>
cudaError_t set_smem_once(Kern k, size_t bytes, int& configured_dev) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_dev != dev) {
        e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
        if (e != cudaSuccess) return e;
        configured_dev = dev;
    }
    return cudaSuccess;
}

template <int T>
cudaError_t launch_decode(const uint32_t* signs, const float* ws, const float* x, float* y, int N, int K, int M,
                          cudaStream_t s) {
    static int configured = -1;
    cudaError_t e = set_smem_once(lut4_decode_kernel<T>, DecLayout<T>::bytes(kDecMaxSlices) + 1024, configured);
    if (e != cudaSuccess) return e;
    const int nbk = K / 32;
    // K slices: about one stage each, at most eight, each a whole number of 4-block quads
    const int nsl = min(kDecMaxSlices, (nbk + kDecStage - 1) / kDecStage);
    const int ks = ((nbk + nsl - 1) / nsl + 3) / 4 * 4;
    const size_t smem = DecLayout<T>::bytes(nsl) + 1024;
    CUtensorMap tmS, tmW;
    if (!make_tmap_2d(&tmS, signs, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, nbk, N, static_cast<uint64_t>(nbk) * 4,
                      kDecStage, 32, true) ||
        !make_tmap_2d(&tmW, ws, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, nbk, N, static_cast<uint64_t>(nbk) * 4,
                      kDecStage, 32, true))
        return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((N + kDecRows - 1) / kDecRows, nsl);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = nsl;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, lut4_decode_kernel<T>, tmS, tmW, x, y, N, K, M, ks);
}

cudaError_t launch_decode_persistent(const uint32_t* signs, const float* ws, const float* x, float* y, int N, int K,
                                     cudaStream_t s) {
    static int configured = -1;
    const int nbk = K / 32;
    const size_t smem = pd_layout(nbk).bytes + 1024;
    cudaError_t e = set_smem_once(lut4_decode_persistent_kernel, pd_layout(kPdMaxBlocks).bytes + 1024, configured);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    CUtensorMap tmS, tmW;
    if (!make_tmap_2d(&tmS, signs, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, nbk, N, static_cast<uint64_t>(nbk) * 4,
                      kPdBoxWords, 32, true) ||
        !make_tmap_2d(&tmW, ws, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, nbk, N, static_cast<uint64_t>(nbk) * 4,
                      kPdBoxWords, 32, true))
        return cudaErrorInvalidValue;
    const int tiles = (N + 31) / 32;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(min(tiles, sms));
    cfg.blockDim = dim3(kPdWarps * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, lut4_decode_persistent_kernel, tmS, tmW, x, y, N, K);
}

template <int MQ>
cudaError_t launch_prefill(const uint32_t* signs, const float* ws, const float* x, float* y, int N, int K, int M,
                           cudaStream_t s) {
    static int configured = -1;
    const size_t smem = pre_smem_bytes<MQ>();
    cudaError_t e = set_smem_once(lut4_prefill_kernel<MQ>, smem, configured);
    if (e != cudaSuccess) return e;
    const dim3 grid((N + kPreRows - 1) / kPreRows, (M + 4 * MQ - 1) / (4 * MQ));
    lut4_prefill_kernel<MQ><<<grid, kPreRows, smem, s>>>(signs, ws, x, y, N, K, M);
    return cudaGetLastError();
}

}  // namespace

GQ_ERROR_ACCESSOR(w1a32)

cudaError_t launch_q1s32_f32(const uint32_t* signs, const float* ws, const float* x, float* y, int M, int N, int K,
                             int path, cudaStream_t s) {
    if (path == GQ_PATH_LUT4) {
        // decode through TMA needs rows of 16-byte multiples (K % 128 == 0) on 16-byte boundaries
        const bool tma_ok = K % 128 == 0 && (reinterpret_cast<uintptr_t>(signs) & 15) == 0 &&
                            (reinterpret_cast<uintptr_t>(ws) & 15) == 0;
        if (M == 1 && tma_ok && K / 32 <= kPdMaxBlocks) return launch_decode_persistent(signs, ws, x, y, N, K, s);
        if (M == 1 && tma_ok) return launch_decode<1>(signs, ws, x, y, N, K, M, s);
        if (M == 2 && tma_ok) return launch_decode<2>(signs, ws, x, y, N, K, M, s);
        if (M <= 4 && tma_ok) return launch_decode<4>(signs, ws, x, y, N, K, M, s);
        if (M <= 4) return launch_prefill<1>(signs, ws, x, y, N, K, M, s);
        if (M <= 8) return launch_prefill<2>(signs, ws, x, y, N, K, M, s);
        if (M <= 16) return launch_prefill<4>(signs, ws, x, y, N, K, M, s);
        return launch_prefill<8>(signs, ws, x, y, N, K, M, s);
    }
    const dim3 grid((N + kRowsPerCta - 1) / kRowsPerCta, M);
    q1s32_f32_gemv_kernel<<<grid, kWarps * 32, 0, s>>>(signs, ws, x, y, N, K);
    return cudaGetLastError();
}

}  // namespace gq
