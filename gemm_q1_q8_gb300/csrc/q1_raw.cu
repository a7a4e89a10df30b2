// Q1_0 x Q8_0 on the pages' own bytes, without the resident repack (browseml-gpu.js: Q1_DOT_WGSL
// reads the 18-byte Q1_0 blocks and 34-byte Q8_0 blocks as stored; packQ8 repacks activations into
// f32 scales and u32 code words).
//
// q1_gemv_raw_kernel: a thread block covers 32 rows and walks the blocks in steps of 8:
//  * the 32 rows x 8 blocks x 18 bytes of the step are staged in shared memory with consecutive
//    16-bit loads (rows are contiguous runs of blocks; any row length, 2-byte alignment);
//  * warp j builds the tables of block j of the step: lane 8k + l holds the 16 exact products
//    d1 * s(nib) of lane group l of sub-block k, s(nib) = sum_c (bit c of nib ? q_c : wrapneg(q_c))
//    over the group's four quants (bit c of the nibble = weight 4l + c of the sub-block, the pages'
//    least-significant-bit-first order);
//  * warp j then forms ab of block j for its 32 rows (lane = row): per sub-block k the row's sign
//    word k, nibble l indexing table (k, l): ab[l] = p (k = 0) or ab[l] + p, rounded to nearest;
//  * warp l of the first eight runs acc[l] = fma(d0, ab[l], acc[l]) over the step's blocks in order;
//  * at the end warp 0 adds each row's eight accumulators in the pages' order.
// The table rows are 17 words apart, so the builders' stores and the 32 lanes' lookups (at most 16
// distinct words of one table) are free of bank conflicts.  The next step's weight and activation
// words are loaded into registers while the current step is summed, so a step costs its work
// rather than a round trip to memory; the kernel is launched as a programmatic dependent, its
// first step's weights requested before the wait for the preceding grids.
#include "gq_internal.cuh"

namespace gq {
namespace {

constexpr int kRawRows = 32;
constexpr int kRawStep = 8;                      // blocks per step (one warp each)
constexpr int kRawHalves = kRawStep * 18 / 2;    // 16-bit words of one row's step (72)
constexpr int kTabStride = 17;
constexpr int kRowPad = kRawHalves + 2;         // 37 words per staged row: the rows' reads hit distinct banks

__global__ void __launch_bounds__(kRawStep * 32)
q1_gemv_raw_kernel(const uint16_t* __restrict__ w, const uint16_t* __restrict__ act, float* __restrict__ y,
                   int rows, int nb) {
    __shared__ __align__(4) uint16_t s_w[kRawRows][kRowPad];
    __shared__ float s_tab[kRawStep][32 * kTabStride];
    __shared__ float s_ab[kRawStep][8][kRawRows];
    __shared__ float s_d0[kRawStep][kRawRows];
    __shared__ float s_acc[8][kRawRows];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = blockIdx.x * kRawRows;
    const size_t row_halves = static_cast<size_t>(nb) * 9;          // 18 bytes per block
    float chain = 0.0f;                                             // warps 0..7: lane group `warp`
    constexpr int kPer = kRawRows * kRawHalves / (kRawStep * 32);   // staged words per thread (9)
    static_assert(kPer * kRawStep * 32 == kRawRows * kRawHalves, "whole words per thread");
    const int k = lane >> 3, l = lane & 7;                          // a table builder's (sub-block, lane)

    // the weight words of step b0 (thread t: items t, t + 256, ...) and the activation words of its
    // table (warp j: block b0 + j)
    uint16_t wn[kPer];
    auto load_w = [&](int b0) {
        const int nbs = min(kRawStep, nb - b0);
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int u = threadIdx.x + i * kRawStep * 32;
            const int r = u / kRawHalves, o = u % kRawHalves;
            wn[i] = (row0 + r < rows && o < nbs * 9) ? w[static_cast<size_t>(row0 + r) * row_halves + b0 * 9 + o]
                                                     : static_cast<uint16_t>(0);
        }
    };
    uint16_t an[3];
    auto load_a = [&](int b0) {
        if (b0 + warp < nb) {
            const uint16_t* blk = act + static_cast<size_t>(4 * (b0 + warp) + k) * 17;    // 34-byte Q8_0 block
            an[0] = blk[0];
            an[1] = blk[1 + 2 * l];
            an[2] = blk[2 + 2 * l];
        }
    };
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    load_w(0);                                                      // weights: before the wait
    asm volatile("griddepcontrol.wait;" ::: "memory");              // the activations are ready
    load_a(0);

    for (int b0 = 0; b0 < nb; b0 += kRawStep) {
        const int nbs = min(kRawStep, nb - b0);
        // stage the step's raw weight words, then request the next step's
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int u = threadIdx.x + i * kRawStep * 32;
            s_w[u / kRawHalves][u % kRawHalves] = wn[i];
        }
        const uint16_t a0 = an[0], a1 = an[1], a2 = an[2];
        if (b0 + kRawStep < nb) {
            load_w(b0 + kRawStep);
            load_a(b0 + kRawStep);
        }
        // tables of block j = warp of the step
        if (warp < nbs) {
            const float d1 = f16_to_f32(a0);
            const uint32_t qw = static_cast<uint32_t>(a1) | (static_cast<uint32_t>(a2) << 16);
            int pos[4], neg[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int q = static_cast<int>(static_cast<int8_t>((qw >> (8 * c)) & 0xFFu));
                pos[c] = q;
                neg[c] = (q == -128) ? -128 : -q;
            }
            float* tab = &s_tab[warp][lane * kTabStride];
#pragma unroll
            for (int nib = 0; nib < 16; ++nib) {
                int s = 0;
#pragma unroll
                for (int c = 0; c < 4; ++c) s += ((nib >> c) & 1) ? pos[c] : neg[c];
                tab[nib] = __fmul_rn(d1, static_cast<float>(s));        // exact: 11 x 10 significant bits
            }
        }
        __syncthreads();
        // ab of block j = warp for the 32 rows (the builders' k, l above name their own item)
        if (warp < nbs) {
            const uint16_t* wr = &s_w[lane][9 * warp];
            const float* tab = s_tab[warp];
            float ab[8];
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint32_t wk = static_cast<uint32_t>(wr[1 + 2 * kk]) | (static_cast<uint32_t>(wr[2 + 2 * kk]) << 16);
#pragma unroll
                for (int ll = 0; ll < 8; ++ll) {
                    const float p = tab[(8 * kk + ll) * kTabStride + ((wk >> (4 * ll)) & 0xFu)];
                    ab[ll] = (kk == 0) ? p : __fadd_rn(ab[ll], p);
                }
            }
#pragma unroll
            for (int ll = 0; ll < 8; ++ll) s_ab[warp][ll][lane] = ab[ll];
            s_d0[warp][lane] = f16_to_f32(wr[0]);
        }
        __syncthreads();
        if (warp < 8) {
#pragma unroll
            for (int j = 0; j < kRawStep; ++j)
                if (j < nbs) chain = __fmaf_rn(s_d0[j][lane], s_ab[j][warp][lane], chain);
        }
        __syncthreads();
    }
    if (warp < 8) s_acc[warp][lane] = chain;
    __syncthreads();
    if (warp == 0 && row0 + lane < rows) {
        // ((a0 + a4) + (a2 + a6)) + ((a1 + a5) + (a3 + a7))
        const float lo = __fadd_rn(__fadd_rn(s_acc[0][lane], s_acc[4][lane]), __fadd_rn(s_acc[2][lane], s_acc[6][lane]));
        const float hi = __fadd_rn(__fadd_rn(s_acc[1][lane], s_acc[5][lane]), __fadd_rn(s_acc[3][lane], s_acc[7][lane]));
        y[row0 + lane] = __fadd_rn(lo, hi);
    }
}

// packQ8: column c's 32-block b -> d[c * nb32 + b] = its f16 scale as f32 (exact), and
// q[(c * nb32 + b) * 8 + v] = its quant bytes 4v..4v+3 as a little-endian word.
__global__ void pack_q8_0_kernel(const uint16_t* __restrict__ raw, long long blocks, float* __restrict__ d,
                                 uint32_t* __restrict__ q) {
    const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= blocks) return;
    const uint16_t* b = raw + i * 17;
    d[i] = f16_to_f32(b[0]);
#pragma unroll
    for (int v = 0; v < 8; ++v)
        q[i * 8 + v] = static_cast<uint32_t>(b[1 + 2 * v]) | (static_cast<uint32_t>(b[2 + 2 * v]) << 16);
}

}  // namespace

cudaError_t launch_q1_gemv_raw(const void* w, const void* act, float* y, int rows, int n, cudaStream_t s) {
    // a programmatic dependent of the previous launch on the stream (see the kernel)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((rows + kRawRows - 1) / kRawRows);
    cfg.blockDim = dim3(kRawStep * 32);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, q1_gemv_raw_kernel, static_cast<const uint16_t*>(w),
                              static_cast<const uint16_t*>(act), y, rows, n / 128);
}

cudaError_t launch_pack_q8_0(const void* raw, int cols, int n, float* d, uint32_t* q, cudaStream_t s) {
    const long long blocks = static_cast<long long>(cols) * (n / 32);
    const int threads = 256;
    pack_q8_0_kernel<<<static_cast<unsigned>((blocks + threads - 1) / threads), threads, 0, s>>>(
        static_cast<const uint16_t*>(raw), blocks, d, q);
    return cudaGetLastError();
}

}  // namespace gq
