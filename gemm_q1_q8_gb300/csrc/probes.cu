// Roofline probes: the machine's own ceilings, measured in the same session as the kernels whose
// fractions are quoted against them (roofline.html: FILL then a read-only pass, best of five after
// a warm-up; web-xpu-ops README, "Performance, measured against the machine's own ceiling").
//
//  * HBM read: gq_probe_fill writes a non-zero pattern, gq_probe_read streams the buffer with
//    16-byte non-allocating loads, eight in flight per thread, and XOR-reduces what it reads into
//    a word the host can read back (so no load is dead).
//  * Issue rates: one thread block of 32 warps per SM runs a long loop of one instruction kind
//    (or an interleaved pair of kinds) on eight independent chains per thread; thread 0 reads
//    the SM clock before and after (between block barriers).  Rate = warp instructions / cycles.
//  * tcgen05 MMA rates: one thread per SM issues a run of MMAs on shared-memory operands into one
//    TMEM accumulator, commits, and waits (bounded) for their completion.
// None of these is on the hot path; bench.py reports them beside the kernels' fractions.
#include "tc_common.cuh"

namespace gq {
namespace {

// ------------------------------------------------------------------------------------------------
// HBM
// ------------------------------------------------------------------------------------------------
__global__ void probe_fill_kernel(uint4* __restrict__ p, size_t n16, uint32_t seed) {
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16; i += stride) {
        const uint32_t h = static_cast<uint32_t>(i) * 0x9E3779B1u + seed;
        p[i] = make_uint4(h | 1u, (h ^ 0xA5A5A5A5u) | 1u, (h * 3u) | 1u, (h + 0x01234567u) | 1u);
    }
}

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__global__ void __launch_bounds__(1024) probe_read_kernel(const uint4* __restrict__ p, size_t n16,
                                                          uint32_t* __restrict__ sink) {
    constexpr int kInFlight = 8;
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    uint32_t x = 0;
    for (; i + (kInFlight - 1) * stride < n16; i += kInFlight * stride) {
        uint4 v[kInFlight];
#pragma unroll
        for (int u = 0; u < kInFlight; ++u) v[u] = ld_stream(p + i + u * stride);
#pragma unroll
        for (int u = 0; u < kInFlight; ++u) x ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
    }
    for (; i < n16; i += stride) {
        const uint4 v = ld_stream(p + i);
        x ^= v.x ^ v.y ^ v.z ^ v.w;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x ^= __shfl_xor_sync(0xffffffffu, x, o);
    if ((threadIdx.x & 31) == 0) atomicXor(sink, x);
}

// ------------------------------------------------------------------------------------------------
// Issue rates
// ------------------------------------------------------------------------------------------------
constexpr int kIssueThreads = 1024;        // 32 warps: 8 per SMSP
constexpr int kIssueChains = 8;            // independent chains per thread
constexpr int kIssueRounds = 4;            // rounds of the eight chains per loop iteration
constexpr int kIssueSmem = 120 * 1024;     // dynamic shared memory requested: one block per SM

__device__ __forceinline__ void op_ffma(float& a, float b, float c) {
    asm volatile("fma.rn.f32 %0, %0, %1, %2;" : "+f"(a) : "f"(b), "f"(c));
}
__device__ __forceinline__ void op_fadd(float& a, float b) { asm volatile("add.rn.f32 %0, %0, %1;" : "+f"(a) : "f"(b)); }
__device__ __forceinline__ void op_ffma2(float2& a, float2 b, float2 c) {
    asm volatile(
        "{\n\t.reg .b64 ra, rb, rc;\n\t"
        "mov.b64 ra, {%0, %1};\n\tmov.b64 rb, {%2, %3};\n\tmov.b64 rc, {%4, %5};\n\t"
        "fma.rn.f32x2 ra, ra, rb, rc;\n\t"
        "mov.b64 {%0, %1}, ra;\n\t}"
        : "+f"(a.x), "+f"(a.y)
        : "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
}
__device__ __forceinline__ void op_fadd2(float2& a, float2 b) {
    asm volatile(
        "{\n\t.reg .b64 ra, rb;\n\t"
        "mov.b64 ra, {%0, %1};\n\tmov.b64 rb, {%2, %3};\n\t"
        "add.rn.f32x2 ra, ra, rb;\n\t"
        "mov.b64 {%0, %1}, ra;\n\t}"
        : "+f"(a.x), "+f"(a.y)
        : "f"(b.x), "f"(b.y));
}
__device__ __forceinline__ void op_dp4a(uint32_t& a, uint32_t b, uint32_t c) {
    asm volatile("dp4a.u32.s32 %0, %1, %2, %0;" : "+r"(a) : "r"(b), "r"(c));
}
__device__ __forceinline__ void op_lop3(uint32_t& a, uint32_t b, uint32_t c) {
    asm volatile("lop3.b32 %0, %0, %1, %2, 0x96;" : "+r"(a) : "r"(b), "r"(c));
}
__device__ __forceinline__ void op_popc(uint32_t& a) { asm volatile("popc.b32 %0, %0;" : "+r"(a)); }
__device__ __forceinline__ void op_prmt(uint32_t& a, uint32_t b) {
    asm volatile("prmt.b32 %0, %0, %1, 0x3175;" : "+r"(a) : "r"(b));
}
__device__ __forceinline__ void op_shf(uint32_t& a, uint32_t b) {
    asm volatile("shf.l.wrap.b32 %0, %0, %1, 5;" : "+r"(a) : "r"(b));
}
__device__ __forceinline__ void op_imad(uint32_t& a, uint32_t b, uint32_t c) {
    asm volatile("mad.lo.u32 %0, %0, %1, %2;" : "+r"(a) : "r"(b), "r"(c));
}
__device__ __forceinline__ void op_shfl(uint32_t& a) {
    asm volatile("shfl.sync.idx.b32 %0, %0, %0, 0x1f, 0xffffffff;" : "+r"(a));
}
// warp-level (legacy) tensor-core MMAs, accumulator in registers
__device__ __forceinline__ void op_mma_f16(float4& d, uint32_t a, uint32_t b) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %4, %4, %4}, {%5, %5}, "
                 "{%0, %1, %2, %3};"
                 : "+f"(d.x), "+f"(d.y), "+f"(d.z), "+f"(d.w)
                 : "r"(a), "r"(b));
}
__device__ __forceinline__ void op_mma_bf16(float4& d, uint32_t a, uint32_t b) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %4, %4, %4}, {%5, %5}, "
                 "{%0, %1, %2, %3};"
                 : "+f"(d.x), "+f"(d.y), "+f"(d.z), "+f"(d.w)
                 : "r"(a), "r"(b));
}
__device__ __forceinline__ void op_mma_e4m3(float4& d, uint32_t a, uint32_t b) {
    asm volatile("mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0, %1, %2, %3}, {%4, %4, %4, %4}, {%5, %5}, "
                 "{%0, %1, %2, %3};"
                 : "+f"(d.x), "+f"(d.y), "+f"(d.z), "+f"(d.w)
                 : "r"(a), "r"(b));
}
__device__ __forceinline__ void op_mma_s8(float4& d, uint32_t a, uint32_t b) {
    int4 t = make_int4(__float_as_int(d.x), __float_as_int(d.y), __float_as_int(d.z), __float_as_int(d.w));
    asm volatile("mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0, %1, %2, %3}, {%4, %4, %4, %4}, {%5, %5}, "
                 "{%0, %1, %2, %3};"
                 : "+r"(t.x), "+r"(t.y), "+r"(t.z), "+r"(t.w)
                 : "r"(a), "r"(b));
    d = make_float4(__int_as_float(t.x), __int_as_float(t.y), __int_as_float(t.z), __int_as_float(t.w));
}
template <int OFF>
__device__ __forceinline__ void op_lds(uint32_t& a, uint32_t saddr) {
    uint32_t v;
    asm volatile("ld.volatile.shared.u32 %0, [%1 + %2];" : "=r"(v) : "r"(saddr), "n"(OFF));
    a ^= v;
}

// one round: eight ops (or four of each kind for a pair), chain j on accumulator j
template <int KIND, int R>
__device__ __forceinline__ void issue_round(uint32_t (&u)[kIssueChains], float (&f)[kIssueChains],
                                            float2 (&g)[kIssueChains], float4 (&m)[kIssueChains], uint32_t saddr) {
    const float2 g1 = make_float2(0.999f, 1.001f), g2 = make_float2(1e-7f, -1e-7f);
    // small operands: f16 2^-6 (0x2400), bf16 2^-6 (0x3C80), e4m3 2^-3 (0x20), s8 1
    constexpr uint32_t kH = 0x24002400u, kBH = 0x3C803C80u, kE = 0x20202020u, kS = 0x01010101u;
#pragma unroll
    for (int j = 0; j < kIssueChains; ++j) {
        constexpr int off = 128 * (R & 7);
        switch (KIND) {
            case GQ_PROBE_FFMA: op_ffma(f[j], 0.999f, 1e-7f); break;
            case GQ_PROBE_FFMA2: op_ffma2(g[j], g1, g2); break;
            case GQ_PROBE_FADD2: op_fadd2(g[j], g2); break;
            case GQ_PROBE_FADD: op_fadd(f[j], 1e-7f); break;
            case GQ_PROBE_DP4A: op_dp4a(u[j], 0x01020304u, 0x7F7F7F7Fu); break;
            case GQ_PROBE_LOP3: op_lop3(u[j], 0x5A5A5A5Au, 0x33333333u); break;
            case GQ_PROBE_POPC: op_popc(u[j]); break;
            case GQ_PROBE_PRMT: op_prmt(u[j], 0x76543210u); break;
            case GQ_PROBE_SHF: op_shf(u[j], 0x12345678u); break;
            case GQ_PROBE_IMAD: op_imad(u[j], 0x01000193u, 0x9E3779B1u); break;
            case GQ_PROBE_SHFL: op_shfl(u[j]); break;
            case GQ_PROBE_LDS: op_lds<off>(u[j], saddr + 4096u * (j & 3)); break;
            case GQ_PROBE_DP4A_FFMA2:
                if (j & 1) op_ffma2(g[j], g1, g2); else op_dp4a(u[j], 0x01020304u, 0x7F7F7F7Fu);
                break;
            case GQ_PROBE_LDS_SHFL:
                if (j & 1) op_shfl(u[j]); else op_lds<off>(u[j], saddr + 4096u * (j & 3));
                break;
            case GQ_PROBE_FFMA_FFMA2:
                if (j & 1) op_ffma2(g[j], g1, g2); else op_ffma(f[j], 0.999f, 1e-7f);
                break;
            case GQ_PROBE_LOP3_DP4A:
                if (j & 1) op_dp4a(u[j], 0x01020304u, 0x7F7F7F7Fu); else op_lop3(u[j], 0x5A5A5A5Au, 0x33333333u);
                break;
            case GQ_PROBE_FADD_FFMA2:
                if (j & 1) op_ffma2(g[j], g1, g2); else op_fadd(f[j], 1e-7f);
                break;
            case GQ_PROBE_LOP3_FFMA2:
                if (j & 1) op_ffma2(g[j], g1, g2); else op_lop3(u[j], 0x5A5A5A5Au, 0x33333333u);
                break;
            case GQ_PROBE_LOP3_POPC:
                if (j & 1) op_popc(u[j]); else op_lop3(u[j], 0x5A5A5A5Au, 0x33333333u);
                break;
            // The A operand is the chain's previous result (bits masked to keep it small and finite),
            // so no operand conversion can be hoisted out of the loop: e4m3 operands are converted in
            // the issuing warp on this GPU, and that cost belongs to the rate.
            case GQ_PROBE_HMMA_F16: op_mma_f16(m[j], (__float_as_uint(m[j].x) & 0x03FF03FFu) | kH, kH); break;
            case GQ_PROBE_HMMA_BF16: op_mma_bf16(m[j], (__float_as_uint(m[j].x) & 0x007F007Fu) | kBH, kBH); break;
            case GQ_PROBE_QMMA_E4M3: op_mma_e4m3(m[j], (__float_as_uint(m[j].x) & 0x07070707u) | kE, kE); break;
            case GQ_PROBE_IMMA_S8: op_mma_s8(m[j], (__float_as_uint(m[j].x) & 0x03030303u) | kS, kS); break;
            case GQ_PROBE_HMMA_MIX:     // mma : lop3 : lop3 : ffma
                if ((j & 3) == 0) op_mma_f16(m[j], (__float_as_uint(m[j].x) & 0x03FF03FFu) | kH, kH);
                else if ((j & 3) == 3) op_ffma(f[j], 0.999f, 1e-7f);
                else op_lop3(u[j], 0x5A5A5A5Au, 0x33333333u);
                break;
            case GQ_PROBE_QMMA_MIX:
                if ((j & 3) == 0) op_mma_e4m3(m[j], (__float_as_uint(m[j].x) & 0x07070707u) | kE, kE);
                else if ((j & 3) == 3) op_ffma(f[j], 0.999f, 1e-7f);
                else op_lop3(u[j], 0x5A5A5A5Au, 0x33333333u);
                break;
            default: break;
        }
    }
}

template <int KIND>
__global__ void __launch_bounds__(kIssueThreads, 1)
probe_issue_kernel(int iters, unsigned long long* __restrict__ cycles, uint32_t* __restrict__ sink) {
    extern __shared__ __align__(16) uint32_t s_buf[];          // 16 KB used by the shared-load kinds
    for (int i = threadIdx.x; i < 4096; i += blockDim.x) s_buf[i] = static_cast<uint32_t>(i) * 2654435761u;
    const uint32_t saddr = smem_u32(s_buf) + 4u * (threadIdx.x & 31);
    uint32_t u[kIssueChains];
    float f[kIssueChains];
    float2 g[kIssueChains];
    float4 m[kIssueChains];
#pragma unroll
    for (int j = 0; j < kIssueChains; ++j) {
        u[j] = threadIdx.x * 7u + j;
        f[j] = 1.0f + j;
        g[j] = make_float2(1.0f + j, 2.0f + j);
        m[j] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
    __syncthreads();
    unsigned long long t0 = 0;
    if (threadIdx.x == 0) t0 = clock64();
#pragma unroll 1
    for (int it = 0; it < iters; ++it) {
        issue_round<KIND, 0>(u, f, g, m, saddr);
        issue_round<KIND, 1>(u, f, g, m, saddr);
        issue_round<KIND, 2>(u, f, g, m, saddr);
        issue_round<KIND, 3>(u, f, g, m, saddr);
    }
    __syncthreads();
    if (threadIdx.x == 0) cycles[blockIdx.x] = clock64() - t0;
    uint32_t x = 0;
#pragma unroll
    for (int j = 0; j < kIssueChains; ++j)
        x ^= u[j] ^ __float_as_uint(f[j]) ^ __float_as_uint(g[j].x) ^ __float_as_uint(g[j].y) ^
             __float_as_uint(m[j].x) ^ __float_as_uint(m[j].y) ^ __float_as_uint(m[j].z) ^ __float_as_uint(m[j].w);
    if (x == 0x5EED5EEDu) sink[0] = x;    // keeps every chain live
}

template <int KIND>
cudaError_t launch_issue(int grid, int iters, unsigned long long* cycles, uint32_t* sink, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(probe_issue_kernel<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kIssueSmem);
    if (e != cudaSuccess) return e;
    probe_issue_kernel<KIND><<<grid, kIssueThreads, kIssueSmem, s>>>(iters, cycles, sink);
    return cudaGetLastError();
}

// ------------------------------------------------------------------------------------------------
// tcgen05 MMA rates
// ------------------------------------------------------------------------------------------------
constexpr int kMmaSmem = 160 * 1024;       // one block per SM (TMEM columns and a clean clock)
constexpr int kMmaTmemCols = 512;          // the accumulator (N <= 256) and, for one kind, A

struct MmaProbeBars {
    uint64_t done;
    uint32_t tmem_base;
};

template <int KIND>
__device__ __forceinline__ void probe_mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
    if (KIND == GQ_PROBE_MMA_F16_TMEM_A) {
        // A from tensor memory: a_desc carries its TMEM address
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
            "r"(static_cast<uint32_t>(a_desc)), "l"(b_desc), "r"(idesc), "r"(accumulate)
            : "memory");
    } else if (KIND == GQ_PROBE_MMA_F16) {
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
            : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
            : "memory");
    }
}

template <int KIND>
__global__ void __launch_bounds__(128, 1)
probe_mma_kernel(int n, int iters, unsigned long long* __restrict__ cycles) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* base = smem_align1024(smem_raw);
    uint8_t* sA = base;                    // 128 rows x 128 bytes
    uint8_t* sB = base + 128 * 128;        // 256 rows x 128 bytes
    MmaProbeBars* bars = reinterpret_cast<MmaProbeBars*>(sB + 256 * 128);
    const int warp = threadIdx.x >> 5;
    // small finite operands: 1/64 in both formats' encodings (bf16 0x3C80, e4m3 0x20)
    const uint32_t fillw = (KIND == GQ_PROBE_MMA_F8) ? 0x20202020u : 0x3C803C80u;
    for (int i = threadIdx.x; i < (128 + 256) * 128 / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(base)[i] = fillw;
    if (threadIdx.x == 0) {
        mbar_init(&bars->done, 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&bars->tmem_base)),
                     "r"(kMmaTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    if (KIND == GQ_PROBE_MMA_F16_TMEM_A) {
        // the A operand's 8 columns: bf16 1/64 in every lane (each warp its 32 lanes)
        uint32_t v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = fillw;
        tc_st32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + 256u, v);
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    if (threadIdx.x == 0) {
        // D f32; A, B bf16 (kind::f16) or e4m3 (kind::f8f6f4, format code 0); both K-major; N, M = 128
        const uint32_t fmt = (KIND == GQ_PROBE_MMA_F8) ? 0u : 1u;
        const uint32_t idesc = (1u << 4) | (fmt << 7) | (fmt << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
                               (static_cast<uint32_t>(128 >> 4) << 24);
        // A from shared memory, or (the TMEM-operand kind) 8 columns of tensor memory after the
        // 256-column accumulator
        const uint64_t ad = (KIND == GQ_PROBE_MMA_F16_TMEM_A) ? static_cast<uint64_t>(tmem + 256u) : smem_desc(sA);
        const uint64_t bd = smem_desc(sB);
        const unsigned long long t0 = clock64();
        for (int i = 0; i < iters; ++i) probe_mma_ss<KIND>(tmem, ad, bd, idesc, i > 0 ? 1u : 0u);
        tc_commit(&bars->done);
        if (!mbar_wait(&bars->done, 0)) {
            report_error(kErrMmaTimeout);
            if (!mbar_wait(&bars->done, 0)) report_error(kErrDrainTimeout);
        }
        cycles[blockIdx.x] = clock64() - t0;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kMmaTmemCols) : "memory");
}

template <int KIND>
cudaError_t launch_mma_probe(int grid, int n, int iters, unsigned long long* cycles, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(probe_mma_kernel<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kMmaSmem);
    if (e != cudaSuccess) return e;
    probe_mma_kernel<KIND><<<grid, 128, kMmaSmem, s>>>(n, iters, cycles);
    return cudaGetLastError();
}

int sm_count(int* out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(out, cudaDevAttrMultiProcessorCount, dev);
    return static_cast<int>(e);
}

int fail(cudaError_t e) {
    if (e == cudaSuccess) return GQ_OK;
    record_cuda_error(static_cast<int>(e));
    return GQ_ECUDA;
}

}  // namespace

GQ_ERROR_ACCESSOR(probes)

}  // namespace gq

using namespace gq;

extern "C" int gq_probe_sm_count(void) {
    int n = 0;
    return sm_count(&n) == 0 ? n : -1;
}

extern "C" int gq_probe_fill(void* buf_device, size_t bytes, uint32_t seed, gq_stream_t stream) {
    if (bytes < 16 || bytes % 16 != 0) return GQ_EINVAL_SHAPE;
    if (!buf_device || (reinterpret_cast<uintptr_t>(buf_device) & 15)) return GQ_EINVAL_PTR;
    int sms = 0;
    const int se = sm_count(&sms);
    if (se != 0) return fail(static_cast<cudaError_t>(se));
    probe_fill_kernel<<<sms * 4, 512, 0, reinterpret_cast<cudaStream_t>(stream)>>>(static_cast<uint4*>(buf_device),
                                                                                 bytes / 16, seed);
    return fail(cudaGetLastError());
}

extern "C" int gq_probe_read(const void* buf_device, size_t bytes, uint32_t* sink_device, int blocks_per_sm,
                             int threads, gq_stream_t stream) {
    if (bytes < 16 || bytes % 16 != 0 || blocks_per_sm < 1 || blocks_per_sm > 32) return GQ_EINVAL_SHAPE;
    if (threads < 32 || threads > 1024 || threads % 32 != 0) return GQ_EINVAL_SHAPE;
    if (!buf_device || !sink_device || (reinterpret_cast<uintptr_t>(buf_device) & 15) ||
        (reinterpret_cast<uintptr_t>(sink_device) & 3))
        return GQ_EINVAL_PTR;
    int sms = 0;
    const int se = sm_count(&sms);
    if (se != 0) return fail(static_cast<cudaError_t>(se));
    probe_read_kernel<<<sms * blocks_per_sm, threads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4*>(buf_device), bytes / 16, sink_device);
    return fail(cudaGetLastError());
}

extern "C" double gq_probe_issue_insts(int kind, int iters) {
    if (kind < 0 || kind >= GQ_PROBE_ISSUE_KINDS || iters < 1) return 0.0;
    return static_cast<double>(kIssueThreads / 32) * iters * kIssueRounds * kIssueChains;
}

extern "C" int gq_probe_issue(int kind, int iters, unsigned long long* cycles_device, uint32_t* sink_device,
                              gq_stream_t stream) {
    if (kind < 0 || kind >= GQ_PROBE_ISSUE_KINDS || iters < 1 || iters > (1 << 24)) return GQ_EINVAL_SHAPE;
    if (!cycles_device || !sink_device || (reinterpret_cast<uintptr_t>(cycles_device) & 7)) return GQ_EINVAL_PTR;
    int sms = 0;
    const int se = sm_count(&sms);
    if (se != 0) return fail(static_cast<cudaError_t>(se));
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    switch (kind) {
#define GQ_PROBE_CASE(K) \
    case K: e = launch_issue<K>(sms, iters, cycles_device, sink_device, s); break;
        GQ_PROBE_CASE(GQ_PROBE_FFMA)
        GQ_PROBE_CASE(GQ_PROBE_FFMA2)
        GQ_PROBE_CASE(GQ_PROBE_FADD2)
        GQ_PROBE_CASE(GQ_PROBE_FADD)
        GQ_PROBE_CASE(GQ_PROBE_DP4A)
        GQ_PROBE_CASE(GQ_PROBE_LOP3)
        GQ_PROBE_CASE(GQ_PROBE_POPC)
        GQ_PROBE_CASE(GQ_PROBE_PRMT)
        GQ_PROBE_CASE(GQ_PROBE_SHF)
        GQ_PROBE_CASE(GQ_PROBE_IMAD)
        GQ_PROBE_CASE(GQ_PROBE_SHFL)
        GQ_PROBE_CASE(GQ_PROBE_LDS)
        GQ_PROBE_CASE(GQ_PROBE_DP4A_FFMA2)
        GQ_PROBE_CASE(GQ_PROBE_LDS_SHFL)
        GQ_PROBE_CASE(GQ_PROBE_FFMA_FFMA2)
        GQ_PROBE_CASE(GQ_PROBE_LOP3_DP4A)
        GQ_PROBE_CASE(GQ_PROBE_FADD_FFMA2)
        GQ_PROBE_CASE(GQ_PROBE_LOP3_FFMA2)
        GQ_PROBE_CASE(GQ_PROBE_HMMA_F16)
        GQ_PROBE_CASE(GQ_PROBE_HMMA_BF16)
        GQ_PROBE_CASE(GQ_PROBE_QMMA_E4M3)
        GQ_PROBE_CASE(GQ_PROBE_IMMA_S8)
        GQ_PROBE_CASE(GQ_PROBE_HMMA_MIX)
        GQ_PROBE_CASE(GQ_PROBE_QMMA_MIX)
        GQ_PROBE_CASE(GQ_PROBE_LOP3_POPC)
#undef GQ_PROBE_CASE
        default: return GQ_EINVAL_SHAPE;
    }
    return fail(e);
}

extern "C" int gq_probe_mma(int kind, int n, int iters, unsigned long long* cycles_device, gq_stream_t stream) {
    if (kind != GQ_PROBE_MMA_F16 && kind != GQ_PROBE_MMA_F8 && kind != GQ_PROBE_MMA_F16_TMEM_A) return GQ_EUNSUPPORTED;
    if (n < 16 || n > 256 || n % 16 != 0 || iters < 1 || iters > 100000) return GQ_EINVAL_SHAPE;
    if (!cycles_device || (reinterpret_cast<uintptr_t>(cycles_device) & 7)) return GQ_EINVAL_PTR;
    int sms = 0;
    const int se = sm_count(&sms);
    if (se != 0) return fail(static_cast<cudaError_t>(se));
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const cudaError_t e = (kind == GQ_PROBE_MMA_F16)   ? launch_mma_probe<GQ_PROBE_MMA_F16>(sms, n, iters, cycles_device, s)
                          : (kind == GQ_PROBE_MMA_F8) ? launch_mma_probe<GQ_PROBE_MMA_F8>(sms, n, iters, cycles_device, s)
                                                      : launch_mma_probe<GQ_PROBE_MMA_F16_TMEM_A>(sms, n, iters, cycles_device, s);
    return fail(e);
}
