// Internal helpers shared by the libgq kernels (sm_103a only).
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "gq.h"

namespace gq {

// --------------------------------------------------------------------------------------------
// Device-side error word: a kernel whose bounded wait runs out ORs a code in and returns.
// --------------------------------------------------------------------------------------------
enum DeviceError : unsigned {
    kErrWaitTimeout = 1u,      // an mbarrier wait on the kernel's own copies exceeded ~1 s
    kErrDrainTimeout = 2u,     // after a timeout, in-flight copies did not land within ~1 s
    kErrMmaTimeout = 4u,       // an MMA/epilogue handshake exceeded ~1 s
};
// Each translation unit with kernels holds its own word (no relocatable device code needed) and
// exposes it through GQ_ERROR_ACCESSOR(unit): gq_device_error() reads and clears them all.
static __device__ unsigned int g_device_error = 0;

__device__ __forceinline__ void report_error(unsigned code) { atomicOr(&g_device_error, code); }

#define GQ_ERROR_ACCESSOR(unit)                                                        \
    unsigned error_read_clear_##unit() {                                               \
        unsigned v = 0, zero = 0;                                                      \
        if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v)) != cudaSuccess) return ~0u; \
        if (v) cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero));                \
        return v;                                                                      \
    }
unsigned error_read_clear_q1();
unsigned error_read_clear_q1_gemv();
unsigned error_read_clear_ternary();
unsigned error_read_clear_prefill_mma();
unsigned error_read_clear_w1a32();
unsigned error_read_clear_probes();
unsigned error_read_clear_block_q8();

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// The first 1024-aligned byte of a dynamic shared-memory array (the launch reserves 1 KB of slack).
// The __shared__ array itself is offset (its address is not rounded as an integer), so the pointer
// stays in the shared address space and accesses through it compile to shared-memory loads and
// stores rather than generic ones with 64-bit address arithmetic.
__device__ __forceinline__ uint8_t* smem_align1024(uint8_t* p) {
    return p + ((1024u - (smem_u32(p) & 1023u)) & 1023u);
}

// --------------------------------------------------------------------------------------------
// mbarrier + bulk asynchronous copies (the TMA engine, untiled form)
// --------------------------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Waits for the phase with the given parity to complete; gives up after ~1 s and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > 1000000000ull) return false;
    }
}
// Global -> shared bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned),
// completing `bytes` transaction bytes on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// --------------------------------------------------------------------------------------------
// Packed f32x2 arithmetic (sm_100+): two independent IEEE binary32 operations, round to
// nearest even, no flush to zero.
// --------------------------------------------------------------------------------------------
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

// a (four unsigned bytes) . b (four signed bytes) + c, exact in 32-bit integers.
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Exact f16 -> f32 (a widening conversion is exact, subnormals included).
__device__ __forceinline__ float f16_to_f32(uint32_t bits16) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16)));
}

// Q8_0 activation quantization of one value (the stated reading: amax over the 32-block,
// d = amax / 127 rounded to nearest, stored as f16 rounded to nearest even; q = round half up of
// x / d with the f32 d, clamped to [-127, 127]; amax = 0 gives q = 0).
__device__ __forceinline__ float q8_0_scale(float amax) { return __fdiv_rn(amax, 127.0f); }
__device__ __forceinline__ int q8_0_quant(float v, float amax, float dd) {
    if (amax == 0.0f) return 0;
    const float vv = __fdiv_rn(v, dd);
    const float fl = floorf(vv);
    const int qi = static_cast<int>(fl) + (__fsub_rn(vv, fl) >= 0.5f ? 1 : 0);
    return max(-127, min(127, qi));
}

// --------------------------------------------------------------------------------------------
// Launch bodies (defined in the per-operation .cu files; arguments already validated).
// --------------------------------------------------------------------------------------------
constexpr int kTileRows = 128;                   // rows per packed Q1_0 tile
constexpr int kChunkBytes = kTileRows * 16 + kTileRows * 2;   // sign bits + d0 per (tile, block)
constexpr int kMaxN = 1 << 20;                   // reduction length limit of the Q1_0 entry points

cudaError_t launch_q1_pack(const void* raw, int rows, int n, void* packed, cudaStream_t s);
cudaError_t launch_q1_gemv(const void* packed, const void* act, float* y, int rows, int n, void* workspace,
                           int act_format, cudaStream_t s);   // act_format: GQ_ACT_Q8_0 or GQ_ACT_F32
size_t gemv_workspace_bytes(int n);
cudaError_t launch_q1_gemv_persistent(const void* packed, const void* act, float* y, int rows, int n, void* workspace,
                                      int act_format, cudaStream_t s);   // q1_gemv.cu
cudaError_t launch_q1s32_f32(const uint32_t* signs, const float* ws, const float* x, float* y, int M, int N, int K,
                             int path, cudaStream_t s);   // path: GQ_PATH_FMA or GQ_PATH_LUT4
cudaError_t launch_q1_gemv_raw(const void* w, const void* act, float* y, int rows, int n, cudaStream_t s);
cudaError_t launch_pack_q8_0(const void* raw, int cols, int n, float* d, uint32_t* q, cudaStream_t s);
cudaError_t launch_q1_gemv_grouped(const gq_gemv_desc* descs, int count, int total_tiles, int* counter,
                                   cudaStream_t s);
int gemv_tiles_for(int rows);
void record_cuda_error(int err);   // makes err what gq_last_cuda_error() reports on this thread
cudaError_t launch_q1_gemm(const void* packed, const void* act, float* y, int rows, int n, int cols,
                           int path, cudaStream_t s);
cudaError_t launch_block_q8(const float* x, const uint32_t* quants, const float* scales, float* y,
                            int m, int k, int n, cudaStream_t s);
cudaError_t launch_ternary(const uint32_t* P, const uint32_t* N, const uint32_t* X, int32_t* y,
                           int rows, int k, int batch, cudaStream_t s);
cudaError_t launch_quantize(const float* x, int m, int k, uint16_t* d, int8_t* q, uint16_t* op,
                            cudaStream_t s);
cudaError_t launch_prefill_lut4(const uint32_t* signs, const float* ws, const uint16_t* xd,
                                const int8_t* xq, float* y, int M, int N, int K, cudaStream_t s);
cudaError_t launch_wq(int bits, const uint32_t* w, const float* scale, const float* x, float* y, int T, int N, int K,
                      cudaStream_t s);   // bits 8: per-row scale; bits 4: per-128-column-group scale
cudaError_t launch_prefill_mma(const uint32_t* signs, const float* ws, const uint16_t* xd,
                               const uint16_t* xq_op, float* y, int M, int N, int K, cudaStream_t s);

}  // namespace gq

// --------------------------------------------------------------------------------------------
// Tiled TMA (cp.async.bulk.tensor) for 2-D row-major tensors.
// --------------------------------------------------------------------------------------------
#include <cuda.h>

namespace gq {

// Encodes a 2-D tiled tensor map: `rows` x `inner` elements of `elem_bytes` bytes, row pitch
// `pitch_bytes` (multiple of 16), box = box_inner x box_rows, 128-byte swizzle when `swizzle128`.
// Out-of-range boxes read as zero.  Returns false if the driver refuses.
bool make_tmap_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, int elem_bytes,
                  uint64_t inner, uint64_t rows, uint64_t pitch_bytes, uint32_t box_inner,
                  uint32_t box_rows, bool swizzle128);

// The same with an explicit swizzle mode.
bool make_tmap_2d_swizzle(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, uint64_t inner,
                          uint64_t rows, uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_rows,
                          CUtensorMapSwizzle swizzle);

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` in a tile written with the 128-byte
// swizzle (rows of 128 bytes, tile base 1024-byte aligned).
__device__ __forceinline__ uint32_t swz128(int row, int chunk) {
    return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}
// The same for the 32-byte swizzle (rows of 32 bytes, tile base 256-byte aligned): address bit 4
// is XORed with bit 7, i.e. the chunk (0 or 1) with bit 2 of the row.
__device__ __forceinline__ uint32_t swz32(int row, int chunk) {
    return static_cast<uint32_t>(row * 32 + ((chunk ^ ((row >> 2) & 1)) << 4));
}

}  // namespace gq
