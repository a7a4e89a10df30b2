// Ternary bitplane GEMV on sm_103a (BonsaiのWebGPUカーネルを読み解く: w = P - N with P/N
// bitplanes, X the binarized activation bitplane, dot = 2*(popc(P&X) - popc(N&X)) - popc(P) +
// popc(N)).
//
// Evaluated as dot = 2*popc((P & X) | (N & ~X)) - popc(P) - popc(N): the two masked sets are
// disjoint when P & N = 0, and a position with both bits set contributes 2 - 2 = 0 either way,
// so this is the same integer for every input -- one LOP3 per word and activation.  The popcounts
// of a chunk row's 32 words are summed through carry-save adders (full adders on whole words, the
// idea of Harley and Seal's popcount): each group of seven words goes through four adders into
// counters of weight 1, 2 and 4, so 32 words take 34 LOP3 and 15 POPC instead of 32 POPC.  POPC
// issues at a quarter of LOP3's rate on a pipe of its own; this split keeps both pipes about
// equally busy (a full adder tree, 60 LOP3 and 6 POPC, left the POPC pipe idle and ran slower).
//
// The result is an integer sum, so K can be cut anywhere without changing it.  A thread block
// covers `rt` rows (a multiple of 16 or 32, sized so that the row tiles fill the GPU once) and up
// to four 1024-bit K chunks: all of its P, N and X chunks are requested at once by TMA (128-byte
// swizzle for P/N: conflict-free 16-byte reads per row), and four groups of rt threads -- one per
// chunk, one thread per row -- count their chunk and add into shared-memory totals.  K beyond four
// chunks goes to more thread blocks of the same rows, which add their totals into y (zeroed on
// the stream first); with K <= 4096 y is written once.
//
// The kernel is launched as a programmatic dependent of the work before it on the stream: it lets
// its own dependents start at once, requests the weight planes P and N (which nothing before it
// writes), and only then waits for the preceding grids before it requests the activation plane X
// and, later, writes y.  In a stream of GEMVs the weights of the next one stream in while the
// current one finishes.
#include "gq_internal.cuh"

namespace gq {
namespace {

constexpr int kWords = 32;                 // words per chunk row (1024 bits, 128 bytes)
constexpr int kChunksPerCta = 4;           // K chunks per thread block, one group of rt threads each
constexpr int kChunkRowBytes = kWords * 4;

struct TernLayout {
    int rt, batch;
    uint32_t p_off, n_off, x_off, red_off, pn_off, bar_off, bytes;
};

// Shared memory of one thread block (offsets from a 1024-aligned base).
__host__ __device__ inline TernLayout tern_layout(int rt, int batch) {
    TernLayout L{rt, batch, 0, 0, 0, 0, 0, 0, 0};
    const uint32_t plane = static_cast<uint32_t>(kChunksPerCta) * rt * kChunkRowBytes;   // 1024-multiple
    L.p_off = 0;
    L.n_off = plane;
    L.x_off = 2 * plane;
    L.red_off = L.x_off + static_cast<uint32_t>(kChunksPerCta) * batch * kChunkRowBytes;
    L.pn_off = L.red_off + static_cast<uint32_t>(batch) * rt * 4;
    L.bar_off = (L.pn_off + static_cast<uint32_t>(rt) * 4 + 7) & ~7u;
    L.bytes = L.bar_off + kChunksPerCta * 8;
    return L;
}

constexpr int kMaxThreads = 512;          // four per row: up to 128 rows, 128 registers

__device__ __forceinline__ uint32_t u4w(const uint4& v, int c) { return c == 0 ? v.x : c == 1 ? v.y : c == 2 ? v.z : v.w; }

// A carry-save adder on 32 bit positions at once: a + b + c = l + 2h in every position.
__device__ __forceinline__ void csa(uint32_t& h, uint32_t& l, uint32_t a, uint32_t b, uint32_t c) {
    h = (a & b) | (a & c) | (b & c);
    l = a ^ b ^ c;
}

// sum over j < NW of popc(word(j)): groups of seven words through four adders (7 -> counters of
// weight 1, 2 and 4: three POPC), then a triple, then single words; about as much POPC issue as
// LOP3 issue, which run on separate pipes
template <int NW, class F>
__device__ __forceinline__ int popc_sum(F word) {
    int c1 = 0, c2 = 0, c4 = 0;
#pragma unroll
    for (int i = 0; i + 7 <= NW; i += 7) {
        uint32_t a1, s1, a2, s2, a3, s, f, t;
        csa(a1, s1, word(i), word(i + 1), word(i + 2));
        csa(a2, s2, word(i + 3), word(i + 4), word(i + 5));
        csa(a3, s, s1, s2, word(i + 6));
        csa(f, t, a1, a2, a3);
        c1 += __popc(s);
        c2 += __popc(t);
        c4 += __popc(f);
    }
    constexpr int r0 = NW - NW % 7;
#pragma unroll
    for (int i = r0; i + 3 <= NW; i += 3) {
        uint32_t h, l;
        csa(h, l, word(i), word(i + 1), word(i + 2));
        c1 += __popc(l);
        c2 += __popc(h);
    }
#pragma unroll
    for (int i = r0 + (NW - r0) / 3 * 3; i < NW; ++i) c1 += __popc(word(i));
    return c1 + 2 * c2 + 4 * c4;
}

__global__ void __launch_bounds__(kMaxThreads)
ternary_kernel(const __grid_constant__ CUtensorMap tmP, const __grid_constant__ CUtensorMap tmN,
               const __grid_constant__ CUtensorMap tmX, int32_t* __restrict__ y, int rows, int k, int batch,
               int rt, int accumulate) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* base = smem_align1024(smem_raw);
    const TernLayout L = tern_layout(rt, batch);
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + L.bar_off);
    int* red = reinterpret_cast<int*>(base + L.red_off);      // [batch][rt]
    int* pnr = reinterpret_cast<int*>(base + L.pn_off);       // [rt]
    const int g = threadIdx.x / rt, r = threadIdx.x - g * rt;
    const int row0 = blockIdx.x * rt;
    const int c0 = blockIdx.y * kChunksPerCta;
    const int chunks = k / (32 * kWords);
    const int nch = min(kChunksPerCta, chunks - c0);
    const uint32_t chunk_bytes = 2u * rt * kChunkRowBytes + static_cast<uint32_t>(batch) * kChunkRowBytes;

    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (threadIdx.x == 0) {
        prefetch_tmap(&tmP);
        prefetch_tmap(&tmN);
        prefetch_tmap(&tmX);
        for (int c = 0; c < nch; ++c) mbar_init(&bars[c], 1);
        fence_barrier_init();
        for (int c = 0; c < nch; ++c) {
            const uint32_t po = static_cast<uint32_t>(c) * rt * kChunkRowBytes;
            mbar_arrive_expect_tx(&bars[c], chunk_bytes);
            tma_load_2d(base + L.p_off + po, &tmP, (c0 + c) * kWords, row0, &bars[c]);
            tma_load_2d(base + L.n_off + po, &tmN, (c0 + c) * kWords, row0, &bars[c]);
        }
        // the activations (and, below, the outputs) only after the preceding grids are done
        asm volatile("griddepcontrol.wait;" ::: "memory");
        for (int c = 0; c < nch; ++c)
            tma_load_2d(base + L.x_off + static_cast<uint32_t>(c) * batch * kChunkRowBytes, &tmX, (c0 + c) * kWords, 0,
                        &bars[c]);
    }
    for (int i = threadIdx.x; i < batch * rt; i += blockDim.x) red[i] = 0;
    for (int i = threadIdx.x; i < rt; i += blockDim.x) pnr[i] = 0;
    __syncthreads();

    // a warp may hold rows of two chunk groups (rt a multiple of 16): after the waits its threads
    // count together
    const bool landed = g < nch && mbar_wait(&bars[g], 0);
    __syncwarp();
    if (g < nch) {
        if (!landed) {
            // let the copy land (bounded) before the thread block can exit
            if (r == 0) {
                report_error(kErrWaitTimeout);
                if (!mbar_wait(&bars[g], 0)) report_error(kErrDrainTimeout);
            }
        } else {
            const uint8_t* Pt = base + L.p_off + static_cast<uint32_t>(g) * rt * kChunkRowBytes;
            const uint8_t* Nt = base + L.n_off + static_cast<uint32_t>(g) * rt * kChunkRowBytes;
            const uint4* Xt =
                reinterpret_cast<const uint4*>(base + L.x_off + static_cast<uint32_t>(g) * batch * kChunkRowBytes);
            // the row's 32 P and N words of this chunk stay in registers for every activation
            uint4 p4[8], n4[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                p4[j] = *reinterpret_cast<const uint4*>(Pt + swz128(r, j));
                n4[j] = *reinterpret_cast<const uint4*>(Nt + swz128(r, j));
            }
            const int pn = popc_sum<64>([&](int j) { return j < 32 ? u4w(p4[j >> 2], j & 3) : u4w(n4[(j - 32) >> 2], j & 3); });
            atomicAdd(&pnr[r], pn);
            for (int b = 0; b < batch; ++b) {
                uint4 x4[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) x4[j] = Xt[b * 8 + j];
                const int cnt = popc_sum<32>([&](int j) {
                    const uint32_t x = u4w(x4[j >> 2], j & 3);
                    return (u4w(p4[j >> 2], j & 3) & x) | (u4w(n4[j >> 2], j & 3) & ~x);
                });
                atomicAdd(&red[b * rt + r], cnt);
            }
        }
    }
    __syncthreads();
    if (g == 0) {
        const int row = row0 + r;
        if (row < rows) {
            for (int b = 0; b < batch; ++b) {
                const int v = 2 * red[b * rt + r] - pnr[r];
                int32_t* dst = y + static_cast<size_t>(b) * rows + row;
                if (accumulate) atomicAdd(dst, v);
                else *dst = v;
            }
        }
    }
}

int sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cached[dev] = n;
    }
    return cached[dev];
}

}  // namespace

GQ_ERROR_ACCESSOR(ternary)

cudaError_t launch_ternary(const uint32_t* P, const uint32_t* N, const uint32_t* X, int32_t* y, int rows, int k,
                           int batch, cudaStream_t s) {
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    const int chunks = k / (32 * kWords);
    const int slices = (chunks + kChunksPerCta - 1) / kChunksPerCta;
    // rows per thread block: the row tiles x K slices fill the GPU about once, within the limits of
    // threads (four per row) and shared memory
    int max_rt = kMaxThreads / kChunksPerCta;
    while (max_rt > 32 && tern_layout(max_rt, batch).bytes + 1024 > 227u * 1024u) max_rt -= 32;
    // rows per block in multiples of 32 (each chunk group whole warps), or of 16 at one activation:
    // there the even split (48-row blocks, 96 rows on every SM for 14,336 rows, against 64-row
    // blocks leaving 128 rows on some SMs) pays, 2.74 -> 2.65 us; with more activations a warp
    // holding rows of two chunk groups waits for the later chunk before it counts (batch 4: 4.27
    // against 3.58 us)
    const int rq = batch == 1 ? 16 : 32;
    // thread blocks per SM: at a few activations the launch is a short fetch-bound wave, and two
    // smaller blocks per SM let one block's counting overlap the other's fetch (batch 1: 3.5 ->
    // 3.1 us; three per SM measured 3.8 us); at batch 16 the popcount work favours one larger block
    const int per_sm = batch <= 4 ? 2 : 1;
    const int want_tiles = per_sm * sms / slices > 0 ? per_sm * sms / slices : 1;
    int rt = ((rows + want_tiles - 1) / want_tiles + rq - 1) / rq * rq;
    if (rt < rq) rt = rq;
    if (rt > max_rt) rt = max_rt;
    const size_t smem = tern_layout(rt, batch).bytes + 1024;

    CUtensorMap tmP, tmN, tmX;
    const uint64_t words = static_cast<uint64_t>(k) / 32;
    if (!make_tmap_2d(&tmP, P, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, words, rows, words * 4, kWords, rt, true) ||
        !make_tmap_2d(&tmN, N, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, words, rows, words * 4, kWords, rt, true) ||
        !make_tmap_2d(&tmX, X, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, words, batch, words * 4, kWords, batch, false))
        return cudaErrorInvalidValue;
    if (slices > 1) {
        const cudaError_t e = cudaMemsetAsync(y, 0, static_cast<size_t>(batch) * rows * sizeof(int32_t), s);
        if (e != cudaSuccess) return e;
    }
    static int configured_dev = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_dev != dev) {
        e = cudaFuncSetAttribute(ternary_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess) return e;
        configured_dev = dev;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((rows + rt - 1) / rt, slices);
    cfg.blockDim = dim3(kChunksPerCta * rt);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, ternary_kernel, tmP, tmN, tmX, y, rows, k, batch, rt, slices > 1 ? 1 : 0);
}

}  // namespace gq
