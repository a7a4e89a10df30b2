/*
 * gq.h -- C ABI of libgq: low-bit block-quantized weight x activation matvec / matmul on GB300
 * (sm_103a).
 *
 * Conventions for every entry point:
 *  - Pointers named *device* point to device memory owned by the caller; the library never
 *    allocates or frees device memory on a call, never synchronizes the stream, and keeps no
 *    per-call state.  Host pointers are named as such.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default stream) and
 *    completes asynchronously.
 *  - Every call validates its arguments on the host before launching anything and returns an
 *    int status: GQ_OK or one of the GQ_E* codes below.  A rejected call launches nothing.
 *    Nothing is truncated silently: a reduction length that is not a whole number of blocks is
 *    an error, not a dropped tail.
 *  - After GQ_ECUDA, gq_last_cuda_error() returns the cudaError_t of the failed launch (per
 *    calling thread).
 *  - Decode kernels are launched as programmatic dependents of the work before them on the stream:
 *    they may start, and read their weights, before that work has finished, and they wait for it
 *    before they read an activation or write an output.  Weights must therefore not be written by
 *    the immediately preceding launch on the stream if that launch signals programmatic completion
 *    early (no launch of this library writes weights; an ordinary kernel or copy is waited for).
 *  - Kernels wait on nothing but their own asynchronous copies, and every such wait is bounded
 *    (about one second).  A wait that runs out sets a device-side error word and the kernel
 *    returns; gq_device_error() reads and clears it.
 *
 * Sources (page title, section) for the operations:
 *  [P1] browseml-gpu.js (browseML / bankML): header comment on the arithmetic; Q1_DOT_WGSL,
 *       Q1_MM_WGSL, Q1_MM4_WGSL; packQ1 / packQ8; gpuMatMul.
 *  [P2] kopitiam-gpu src/shaders/block_q8_matmul_nt.wgsl: header (bindings, PACKING,
 *       ACCUMULATION ORDER), fn quant_at, fn main.
 *  [P3] BonsaiのWebGPUカーネルを読み解く: the ternary P/N bitplane popcount identity; the
 *       decode / prefill kernel figure (q1_bits + q1_scales, binary-lut4-matmul LUT4 prefill,
 *       subgroup-matrix third path).
 */
#ifndef GQ_H
#define GQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* gq_stream_t;   /* the same type as cudaStream_t */

enum gq_status {
    GQ_OK = 0,
    GQ_EINVAL_SHAPE = 1,   /* a size is <= 0, too large, or not a whole number of blocks  */
    GQ_EINVAL_PTR = 2,     /* a required pointer is NULL or not aligned as documented     */
    GQ_EUNSUPPORTED = 3,   /* the requested path does not exist for this operation/shape  */
    GQ_ECUDA = 4           /* a CUDA launch failed; see gq_last_cuda_error()               */
};

enum gq_path {
    GQ_PATH_AUTO = 0,      /* the library picks by shape                                    */
    GQ_PATH_DP4A = 1,      /* integer dot products (dp4a) on the CUDA cores                 */
    GQ_PATH_LUT4 = 2,      /* 16-entry subset-sum tables per 4 activations, nibble lookups  */
    GQ_PATH_MMA = 3,       /* tcgen05 tensor-core MMA (kind::f16) with a fixed-order epilogue */
    GQ_PATH_FMA = 4        /* weights expanded to +-1.0 and multiply-added on the CUDA cores  */
};

/* Library version string (static storage). */
const char* gq_version(void);
/* Human-readable name of a status code (static storage). */
const char* gq_status_string(int status);
/* cudaError_t of the last failed launch on this host thread (0 if none). */
int gq_last_cuda_error(void);
/* Reads and clears the device-side error word of the current device: 0 if no kernel has
 * reported a timed-out wait since the last call, else a nonzero code.  Synchronizes the device. */
int gq_device_error(void);

/* ============================================================================================
 * Q1_0 weights x Q8_0 activations  [P1]
 *
 * Q1_0 block (18 bytes, the pages' storage): f16 d0 (little-endian) then 128 sign bits; weight
 * j = 32k + e of the block is bit e%8 of byte 2 + 4k + e/8 (bit 1 -> +q, bit 0 -> -q).
 * Q8_0 block (34 bytes): f16 d1 (little-endian) then 32 int8 quants.
 * A row of n weights is n/128 Q1_0 blocks; an activation vector of n values is n/32 Q8_0 blocks;
 * Q1_0 block i pairs with Q8_0 blocks 4i..4i+3.
 *
 * Result per (row, activation) -- the pages' exact operation order, reproduced bit for bit:
 *   per block i, sub-block k = 0..3, lane l = 0..7 (weights 4l..4l+3 of the sub-block):
 *     s = sum (bit ? q : -q), the negate wrapping as int8 (-(-128) = -128)
 *     p = d1 * s (exact), ab[l] = p (k = 0) or ab[l] + p (k > 0)   (round to nearest even)
 *     acc[l] = fma(d0, ab[l], acc[l])                                 (correctly rounded)
 *   y = ((acc0+acc4)+(acc2+acc6)) + ((acc1+acc5)+(acc3+acc7)), acc from +0.
 * ========================================================================================== */

/* Bytes of the packed (resident) form of a rows x n Q1_0 matrix; 0 if the shape is invalid. */
size_t gq_q1_0_packed_bytes(int rows, int n);

/* One-time repack of Q1_0 weights into the kernels' resident layout ([P1] packQ1: "repacked
 * once"; the engine keeps weights resident).
 *   raw_device    rows * (n/128) * 18 bytes, the pages' AoS blocks, row-major; any alignment.
 *   packed_device gq_q1_0_packed_bytes(rows, n) bytes, 16-byte aligned; fully written
 *                 (rows are padded to a multiple of 128 with zero blocks).
 * Layout (private to the library; treat as opaque): 128-row tiles; per (tile, block) a 2304-byte
 * chunk of 128 x 16 bytes of sign bits (bit-permuted within each 32-bit word) then 128 f16 d0.
 * Errors: GQ_EINVAL_SHAPE if rows < 1, n < 128, n % 128 != 0 or n > 2^20;
 *         GQ_EINVAL_PTR if a pointer is NULL or packed_device is not 16-byte aligned. */
int gq_q1_0_pack(const void* raw_device, int rows, int n, void* packed_device, gq_stream_t stream);

/* Bytes of workspace one decode GEMV needs for an activation of n values: the activation's
 * per-32-value constants (96 bytes per 32 values), built by the call itself, and a 16-byte tile
 * counter. */
size_t gq_q1_q8_workspace_bytes(int n);

/* Decode GEMV ([P1] Q1_DOT_WGSL semantics): y[r] for r < rows.
 *   packed_w_device from gq_q1_0_pack(rows, n); act_device: n/32 Q8_0 blocks (34 bytes each,
 *   2-byte aligned); y_device: rows f32; workspace_device: gq_q1_q8_workspace_bytes(n) bytes,
 *   16-byte aligned, which the call may overwrite.  A matrix with fewer 128-row tiles than the
 *   GPU has SMs takes one launch that builds the activation's constants itself and leaves the
 *   workspace untouched; a larger one takes two launches on `stream` (the constants into the
 *   workspace, then the GEMV, which hands 128-row tiles to its warps through a counter at the
 *   end of the workspace).  Calls that share a workspace must not overlap on the GPU.
 * Errors: as gq_q1_0_pack, plus GQ_EINVAL_PTR if act_device is odd, y_device not 4-aligned or
 * the workspace NULL or not 16-aligned. */
int q1_q8_gemv(const void* packed_w_device, const void* act_device, float* y_device,
               int rows, int n, void* workspace_device, gq_stream_t stream);

/* Activation formats of the decode GEMV (gq_gemv_desc.act_format). */
enum gq_act_format {
    GQ_ACT_Q8_0 = 0,       /* n/32 Q8_0 blocks of 34 bytes (f16 d, 32 int8), 2-byte aligned       */
    GQ_ACT_F32 = 1         /* n f32 values, 16-byte aligned, quantized to Q8_0 inside the call     */
};

/* The decode GEMV over f32 activations, with the Q8_0 quantization of the activations fused into
 * the GEMV's activation-constant step (no separate quantize launch, no Q8_0 round trip through
 * memory).  The result is bit-identical to gq_quantize_q8_0 on x followed by q1_q8_gemv: each
 * 32-block is quantized as that call states (d = f16(amax / 127), q = round half up of x / d
 * with the f32 d, clamped to [-127, 127]; an all-zero block gives d = 0, q = 0).  The pages do
 * not describe a decode-side quantizer; this is the reading of the prefill one.
 *   x_device: n f32, 16-byte aligned; other arguments and launches as q1_q8_gemv.
 * Errors: as q1_q8_gemv, with GQ_EINVAL_PTR if x_device is NULL or not 16-aligned. */
int q1_q8_gemv_f32(const void* packed_w_device, const float* x_device, float* y_device, int rows, int n,
                   void* workspace_device, gq_stream_t stream);

/* Decode GEMV on the pages' own bytes, with no repack of the weights ([P1] Q1_DOT_WGSL reads the
 * 18-byte Q1_0 blocks as stored): the same result as gq_q1_0_pack followed by q1_q8_gemv, bit for
 * bit, for callers that keep their weights in the pages' layout.  Slower than the resident layout
 * (its sign bits are looked up by nibble in tables of the block's exact products d1 * s, built per
 * thread block and 32 rows).
 *   w_q1_0_device: rows * (n/128) * 18 bytes, the pages' AoS blocks, row-major, 2-byte aligned;
 *   act_device: n/32 Q8_0 blocks (34 bytes), 2-byte aligned; y_device: rows f32, 4-byte aligned.
 *   One launch on `stream`; no workspace.
 * Errors: GQ_EINVAL_SHAPE if rows < 1, n < 128, n % 128 != 0 or n > 2^20; GQ_EINVAL_PTR for a
 * NULL or misaligned pointer; GQ_ECUDA. */
int q1_q8_gemv_raw(const void* w_q1_0_device, const void* act_device, float* y_device, int rows, int n,
                   gq_stream_t stream);

/* [P1] packQ8: `cols` activation vectors of n values, each n/32 Q8_0 blocks of 34 bytes (vector
 * after vector, 2-byte aligned), repacked into d_device[c * n/32 + b] = the block's f16 scale as f32
 * (exact) and q_device[(c * n/32 + b) * 8 + v] = its quant bytes 4v..4v+3 as one little-endian word
 * (both 4-byte aligned).  The library's GEMV and GEMM read the 34-byte blocks directly; this is the
 * pages' layout for callers that keep activations in it.
 * Errors: GQ_EINVAL_SHAPE if cols < 1, n < 32, n % 32 != 0 or n > 2^20; GQ_EINVAL_PTR; GQ_ECUDA. */
int gq_pack_q8_0(const void* raw_q8_0_device, int cols, int n, float* d_device, uint32_t* q_device,
                 gq_stream_t stream);

/* Largest n that q1_q8_gemv_noalloc accepts. */
#define GQ_NOALLOC_MAX_N 16384

/* The decode GEMV for callers that cannot allocate device memory (code running inside another
 * allocator's arena, plugins handed raw pointers, paths where an allocation could block or fail):
 * the same result as q1_q8_gemv, bit for bit, with the workspace taken from a fixed block of
 * device memory built into the library (about 48 KB, held by every GPU that loads the library
 * until the process exits).  The pages describe no such variant.
 *   Arguments as q1_q8_gemv without the workspace; n <= GQ_NOALLOC_MAX_N.
 *   The first call on each device looks up that block's address (cudaGetSymbolAddress, with the
 *   device current) and keeps it: make that first call before any stream capture on the device,
 *   and do not reset the device (cudaDeviceReset) between calls.
 *   Every call shares the block, so calls whose work overlaps on the GPU (other streams, other
 *   host threads) race: issue them one after another.  The call itself clears what must start
 *   at zero.  It calls no allocator (no cudaMalloc / cudaFree, no library that allocates).
 * Errors: GQ_EINVAL_SHAPE for rows < 1, n < 128, n % 128 != 0 or n > GQ_NOALLOC_MAX_N;
 *         GQ_EINVAL_PTR as q1_q8_gemv; GQ_ECUDA if the address lookup or a launch fails. */
int q1_q8_gemv_noalloc(const void* packed_w_device, const void* act_device, float* y_device, int rows,
                       int n, gq_stream_t stream);

/* One matrix of a grouped GEMV sweep (all fields filled by the caller except tile_begin). */
typedef struct gq_gemv_desc {
    const void* packed_w;    /* device, from gq_q1_0_pack(rows, n)                      */
    const void* act;         /* device, n/32 Q8_0 blocks, or n f32 (act_format)         */
    float* y;                /* device, rows f32                                        */
    void* workspace;         /* device, gq_q1_q8_workspace_bytes(n), 16-aligned, its own */
    int rows;
    int n;
    int tile_begin;          /* filled by gq_gemv_group_plan                            */
    int act_format;          /* GQ_ACT_Q8_0 (0) or GQ_ACT_F32 (quantized in the call)   */
} gq_gemv_desc;

/* Host-side planning for q1_q8_gemv_grouped: validates every descriptor (host array), sorts the
 * array by n, largest first (stable; each entry keeps its own pointers, so results are
 * unaffected), and fills tile_begin (a prefix sum of 128-row tiles).  *total_tiles receives the
 * number of tiles of the whole group.
 * Errors: GQ_EINVAL_SHAPE / GQ_EINVAL_PTR as q1_q8_gemv for the first bad descriptor (the array
 * is then left unsorted), or GQ_EINVAL_SHAPE if count < 1, count > 65535 or the group exceeds
 * 2^31-1 tiles. */
int gq_gemv_group_plan(gq_gemv_desc* descs_host, int count, int* total_tiles);

/* Grouped decode GEMV: every matrix of a layer stack (e.g. one decode token's sweep) in two
 * launches (all activations' constants, then one persistent GEMV over every tile of the group,
 * which hands 128-row tiles to warps through *counter_device, largest matrix first).
 * descs_device is a device copy of the planned array (count entries, 8-byte aligned);
 * total_tiles is the value gq_gemv_group_plan returned; counter_device is one int of device
 * memory (4-aligned) that the call resets and uses -- calls sharing it, or sharing a
 * descriptor's workspace, must not overlap on the GPU.  Results are bit-identical to calling
 * q1_q8_gemv on each entry.  The host cannot re-validate device descriptors: pass only arrays
 * that gq_gemv_group_plan accepted, unchanged. */
int q1_q8_gemv_grouped(const gq_gemv_desc* descs_device, int count, int total_tiles, int* counter_device,
                       gq_stream_t stream);

/* Bonsai 1-bit weights times f32 activations ([P3] decode/prefill figure: the decode kernel
 * llama-decode-q1-proj.wgsl and the prefill kernel binary-lut4-matmul.wgsl):
 *   y[m * N + n] = sum_b wscale[n * K/32 + b] * sum_t s(n, 32 b + t) * x[m * K + 32 b + t]
 * with s = +1.0 where bit t of signs[n * K/32 + b] is set, -1.0 where it is clear (the same
 * weight arrays as q1s32_q8_gemm).  The page does not fix the order of the float operations, so
 * neither path is defined bit for bit; each result lies within c * 2^-24 * sum_b |wscale| *
 * sum_t |x| of the exact value, c = 32 + ceil(nb/8) for LUT4 at M <= 4 with K % 128 == 0,
 * c = 12 + nb for the other LUT4 cases and c = 40 + ceil(nb/32) for FMA (nb = K/32).  Results are
 * deterministic: the same inputs and path give the same bits on every call.
 *   path GQ_PATH_FMA: the decode formulation -- signs expanded to +-1, each block summed in
 *        order, acc = fma(scale, block_sum, acc), lanes added by a butterfly.
 *   path GQ_PATH_LUT4: per token and 4 activations a table of the 16 signed sums, indexed by the
 *        weight nibble; block sum = the 8 lookups in order; acc = fma(scale, block_sum, acc).
 *   path GQ_PATH_AUTO: LUT4.
 *   signs_device: N * K/32 u32; wscale_device: N * K/32 f32 (both 4-byte aligned; rows that
 *   start on 16 bytes are read with 16-byte loads); x_device: M * K f32, 16-byte aligned;
 *   y_device: M * N f32, 4-byte aligned.  One launch on `stream`; no workspace.
 * Errors: GQ_EINVAL_SHAPE unless N >= 1, 1 <= M <= 65535, 32 <= K <= 65536 and K % 32 == 0;
 *         GQ_EUNSUPPORTED for another path; GQ_EINVAL_PTR for a NULL or misaligned pointer;
 *         GQ_ECUDA. */
int q1s32_f32_gemm(const uint32_t* signs_device, const float* wscale_device, const float* x_device,
                   float* y_device, int M, int N, int K, int path, gq_stream_t stream);

/* q1s32_f32_gemm on the tensor cores (the prefill path; same operation and weight arrays).  The
 * activations are split exactly into three bf16 parts (hi = bf16(x), mid = bf16(x - hi),
 * lo = bf16(x - hi - mid), each rounded to nearest; hi + mid + lo = x for normal x) in the
 * workspace; the tensor cores form each 32-block's p = sum_t s * x (the +-1 weights are exact in
 * bf16), and acc = fma(wscale, p, acc) runs in block order.  The result lies within
 * c * 2^-24 * sum_b |wscale| * sum_t |x| of the exact value with c = nb + 16 (nb = K/32: one fma
 * per block, two units for each of the six tensor-core steps of a block, whose f32 accumulation
 * rounding is not published), and the same inputs give the same bits on every call.
 *   workspace_device: gq_q1s32_mma_workspace_bytes(M, K) bytes (3 * M * K bf16), 16-byte aligned,
 *   overwritten; signs_device 16-byte and wscale_device 8-byte aligned; x_device 4-byte aligned.
 *   Two launches on `stream` (the split, then the prefill MMA kernel).
 * Errors: GQ_EINVAL_SHAPE unless N >= 1, 1 <= M <= 65535 * 128, 64 <= K <= 65536 and K % 64 == 0;
 *         GQ_EINVAL_PTR for a NULL or misaligned pointer; GQ_ECUDA. */
size_t gq_q1s32_mma_workspace_bytes(int M, int K);     /* 0 for an invalid shape */
int q1s32_f32_gemm_mma(const uint32_t* signs_device, const float* wscale_device, const float* x_device,
                       float* y_device, int M, int N, int K, void* workspace_device, gq_stream_t stream);

/* Block-quantized weights times f32 activations (web-xpu-ops README: the op table rows
 * matvecQ8 / matmulQ8 and matvecQ4G128 / matmulQ4G128, and "The q4 format"):
 *   matvec_q8 / matmul_q8 (W8A32, per-row scale):
 *     code k of row n = byte (k % 4) of w[n * K/4 + k/4], least-significant byte first, signed;
 *     y[t * N + n] = scale[n] * sum_k code(n, k) * x[t * K + k].
 *   matvec_q4g128 / matmul_q4g128 (W4A32, one scale per 128 columns):
 *     code k of row n = nibble (k % 8) of w[n * K/8 + k/8], least-significant nibble first,
 *     4-bit two's complement (the page's quantizer emits [-7, 7]; a raw 0x8 reads as -8);
 *     y[t * N + n] = sum_g scale[n * ceil(K/128) + g] * sum_{k in g} code(n, k) * x[t * K + k].
 * The matvec is the matmul with T = 1.  The page fixes no float order, so the results are not
 * defined bit for bit; each lies within c * 2^-24 * sum |scale * code * x| of the exact value
 * (T <= 4: c = 16 * ceil(K/4096) + 10 for 8 bits, c = 28 + ceil(K/512) for 4 bits; T > 4:
 * c = K + 2), and the same inputs give the same bits on every call.
 *   w_device: N * K/4 (8 bits) or N * K/8 (4 bits) u32, 16-byte aligned; scale_device: N (8 bits)
 *   or N * ceil(K/128) (4 bits) f32; x_device: T * K f32, 16-byte aligned; y_device: T * N f32.
 *   One launch on `stream`; no workspace.
 * Errors: GQ_EINVAL_SHAPE unless N >= 1, 1 <= T <= 65535 * 128, 32 <= K <= 65536 and
 *         K % 32 == 0; GQ_EINVAL_PTR for a NULL or misaligned pointer; GQ_ECUDA. */
int matvec_q8(const uint32_t* w_device, const float* scale_device, const float* x_device, float* y_device,
              int N, int K, gq_stream_t stream);
int matmul_q8(const uint32_t* w_device, const float* scale_device, const float* x_device, float* y_device,
              int T, int N, int K, gq_stream_t stream);
int matvec_q4g128(const uint32_t* w_device, const float* scale_device, const float* x_device, float* y_device,
                  int N, int K, gq_stream_t stream);
int matmul_q4g128(const uint32_t* w_device, const float* scale_device, const float* x_device, float* y_device,
                  int T, int N, int K, gq_stream_t stream);

/* matmul_q8 / matmul_q4g128 on the tensor cores (same operations and code layouts as above).  Each
 * activation x is split exactly into three bf16 parts (hi = bf16(x), mid = bf16(x - hi),
 * lo = bf16(x - hi - mid), each rounded to nearest; hi + mid + lo == x for normal x), the int8
 * codes are exact in bf16, and the tensor cores accumulate the code * part products of one
 * 128-column round (three parts x 128 columns) into an f32 partial; 8 bits: the partials are added
 * in f32 with round to nearest, round after round, and y = scale[n] * sum; 4 bits: acc =
 * fma(scale[n, g], partial, acc) round after round (round g is group g), y = acc.  The result lies
 * within c * 2^-24 * sum |scale * code * x| of the exact value with c = ceil(K/128) + 56 (two units
 * per tensor-core step, whose f32 accumulation rounding is not published), and the same inputs
 * give the same bits on every call.  Activations below 2^-126 * 2^16 in magnitude may lose their lowest bits
 * (the residual planes are bf16, whose exponent range is f32's).
 *   workspace_device: gq_wq_mma_workspace_bytes(T, K) bytes (3 * T * K bf16), 16-byte aligned,
 *   overwritten; the other arguments as matmul_q8 / matmul_q4g128.  Two launches on `stream` (the split, then the
 *   tensor-core kernel).
 * Errors: GQ_EINVAL_SHAPE unless N >= 1, 1 <= T <= 65535 * 128, 64 <= K <= 65536 and K % 32 == 0;
 *         GQ_EINVAL_PTR for a NULL or misaligned pointer; GQ_ECUDA. */
size_t gq_wq_mma_workspace_bytes(int T, int K);     /* 0 for an invalid shape */
int matmul_q8_mma(const uint32_t* w_device, const float* scale_device, const float* x_device, float* y_device,
                  int T, int N, int K, void* workspace_device, gq_stream_t stream);
int matmul_q4g128_mma(const uint32_t* w_device, const float* scale_device, const float* x_device, float* y_device,
                      int T, int N, int K, void* workspace_device, gq_stream_t stream);

/* Prefill GEMM over `cols` Q8_0 activation vectors ([P1] Q1_MM_WGSL / Q1_MM4_WGSL): every
 * (row, column) is the GEMV chain above, stored at y[c * rows + r].
 *   act_device: cols * (n/32) Q8_0 blocks, column after column (2-byte aligned).
 *   path: GQ_PATH_DP4A, GQ_PATH_LUT4 or GQ_PATH_AUTO (DP4A); GQ_PATH_MMA -> GQ_EUNSUPPORTED
 *         (the per-4-weight lane sums of this format leave a tensor core nothing dense to do).
 * Errors: as q1_q8_gemv, plus GQ_EINVAL_SHAPE if cols < 1. */
int q1_q8_gemm(const void* packed_w_device, const void* act_device, float* y_device,
               int rows, int n, int cols, int path, gq_stream_t stream);

/* ============================================================================================
 * block_q8_matmul_nt  [P2]:  y = x . w^T with w block-scaled int8.
 *   x_device      [m, k] f32 row-major (4-byte aligned)
 *   quants_device k*n int8 packed four per u32, little-endian: element t of weight row `col` is
 *                 byte (t%4) of word (col*k + t)/4, sign-extended (16-byte aligned)
 *   scales_device [n, k/32] f32
 *   y_device      [m, n] f32 row-major
 * Order (bit for bit): per (row, col), for block b ascending: block_sum = 0; for t < 32:
 * block_sum = block_sum + x*q (a rounded multiply, then a rounded add); acc = acc +
 * scale*block_sum (the same); acc from +0.
 * Errors: GQ_EINVAL_SHAPE if m, k or n < 1, k % 32 != 0, k > 65536 or m > 65535;
 *         GQ_EINVAL_PTR for NULL or misaligned pointers. */
int block_q8_matmul_nt(const float* x_device, const uint32_t* quants_device,
                       const float* scales_device, float* y_device, int m, int k, int n,
                       gq_stream_t stream);

/* ============================================================================================
 * Ternary bitplane GEMV  [P3]:  weights w in {-1, 0, +1} as bitplanes P (w = +1) and N (w = -1),
 * activations binarized to a bitplane X (bit 1 -> +1, bit 0 -> -1); bit j of word v is element
 * 32v + j.  Per (batch b, row r), exactly:
 *   y = 2 * (sum popc(P & X) - sum popc(N & X)) - sum popc(P) + sum popc(N).
 * A position with both P and N set counts as weight 0.
 *   P_device, N_device [rows, k/32] u32 (16-byte aligned); X_device [batch, k/32] u32
 *   (16-byte aligned); y_device [batch, rows] int32.
 * Errors: GQ_EINVAL_SHAPE if rows or batch < 1, k < 1024, k % 1024 != 0 (tiles of 32 words),
 *         k > 65536 or batch > 64;
 *         GQ_EINVAL_PTR for NULL or misaligned pointers. */
int ternary_bitplane_gemv(const uint32_t* P_device, const uint32_t* N_device,
                          const uint32_t* X_device, int32_t* y_device, int rows, int k,
                          int batch, gq_stream_t stream);

/* ============================================================================================
 * Batched prefill with Bonsai-format 1-bit weights  [P3] and Q8_0 activations.
 *
 * Activation quantizer (the pages give none for Q8_0 blocks; the reading is stated here):
 * per 32-block of a row of x, amax = max |x|; d = amax / 127 (round to nearest); the stored
 * scale is f16(d) rounded to nearest even; q = clamp(floor(v) + (v - floor(v) >= 0.5), -127,
 * 127) with v = x / d (round to nearest, the f32 d); amax == 0 gives d = 0 and q = 0.
 *   x_device [m, k] f32; d_device [m, k/32] f16 bits; q_device [m, k] int8 (16-byte aligned);
 *   mma_operand_device: NULL, or [3, m, k] bf16 (16-byte aligned) receiving the operand
 *   q1s32_q8_gemm's MMA path reads: pv = f16(d) * q (exact) split into three bf16 parts,
 *   hi = bf16(pv), mid = bf16(pv - hi), lo = bf16(pv - hi - mid) (each rounded to nearest, so
 *   hi + mid + lo = pv), plane p at offset p * m * k, with the elements of each 32-block
 *   interleaved (position 2u <- element u, 2u+1 <- element u+16).
 * Errors: GQ_EINVAL_SHAPE if m or k < 1, k % 32 != 0 or k > 65536; GQ_EINVAL_PTR. */
int gq_quantize_q8_0(const float* x_device, int m, int k, uint16_t* d_device, int8_t* q_device,
                     uint16_t* mma_operand_device, gq_stream_t stream);

/* Prefill GEMM: y[m, n] = sum over 32-blocks b ascending of
 *     S = sum_t (sign bit ? q : -q) (int8-wrapping negate), p = f16(xd[m,b]) * S (exact),
 *     acc = fma(w_scale[n, b], p, acc) (correctly rounded), acc from +0.
 *   signs_device   [N, K/32] u32, bit t of word b = weight 32b+t, 1 -> +1 (16-byte aligned)
 *   wscale_device  [N, K/32] f32 (4-byte aligned; 8-byte aligned for GQ_PATH_MMA)
 *   xd_device      [M, K/32] f16 bits (4-byte aligned), xq_device [M, K] int8 (16-byte aligned)
 *   xq_mma_device  the three-plane bf16 operand from gq_quantize_q8_0 (required for
 *                  GQ_PATH_MMA, else may be NULL), made from the same d and q as xd_device and
 *                  xq_device, all q in [-127, 127] (as the quantizer produces).  The tensor
 *                  cores form p = f16(d) * S itself: every term and partial sum is a multiple of
 *                  the ulp of f16(d) below 2^12 f16(d), so its f32 accumulation is exact.
 *   y_device       [M, N] f32 row-major
 *   path: GQ_PATH_LUT4, GQ_PATH_MMA, or GQ_PATH_AUTO (MMA when M >= 64 and the operand is
 *   given, else LUT4).  Both paths are bit-identical to the order above.
 * Errors: GQ_EINVAL_SHAPE if M, N or K < 1, K % 64 != 0 or K > 65536; GQ_EUNSUPPORTED for an
 * unknown path or GQ_PATH_DP4A; GQ_EINVAL_PTR for NULL/misaligned pointers (xq_mma_device NULL
 * with GQ_PATH_MMA included). */
int q1s32_q8_gemm(const uint32_t* signs_device, const float* wscale_device,
                  const uint16_t* xd_device, const int8_t* xq_device,
                  const uint16_t* xq_mma_device, float* y_device, int M, int N, int K, int path,
                  gq_stream_t stream);

/* ============================================================================================
 * Roofline probes (measurement only; no hot-path entry point uses them).  The machine's own
 * ceilings, measured in the same session as the kernels whose fractions are quoted against them:
 * roofline.html's read-only bandwidth method (FILL a buffer with a non-zero pattern, then read it
 * with every load live, best of five after a warm-up) and the web-xpu-ops README's "Performance,
 * measured against the machine's own ceiling".
 * ========================================================================================== */

/* Number of SMs of the current device, or -1. */
int gq_probe_sm_count(void);

/* Writes a non-zero pattern derived from `seed` over `bytes` (a multiple of 16) of buf_device
 * (16-byte aligned).  One launch on `stream`.
 * Errors: GQ_EINVAL_SHAPE, GQ_EINVAL_PTR, GQ_ECUDA. */
int gq_probe_fill(void* buf_device, size_t bytes, uint32_t seed, gq_stream_t stream);

/* One read-only pass over `bytes` of buf_device with 16-byte loads that bypass L1 (eight in
 * flight per thread, grid-stride over blocks_per_sm x SMs blocks of `threads` threads), XOR of
 * everything read folded into *sink_device (one u32, 4-byte aligned, which the caller zeroes).
 * The caller times the launch; bytes / time is the read bandwidth.  Use a buffer several times
 * the L2 size.  Errors: GQ_EINVAL_SHAPE unless bytes is a positive multiple of 16,
 * 1 <= blocks_per_sm <= 32 and threads is a multiple of 32 in [32, 1024]; GQ_EINVAL_PTR. */
int gq_probe_read(const void* buf_device, size_t bytes, uint32_t* sink_device, int blocks_per_sm, int threads,
                  gq_stream_t stream);

/* Instruction kinds of gq_probe_issue: one kind alone, or two interleaved one to one. */
enum gq_probe_kind {
    GQ_PROBE_FFMA = 0,          /* fma.rn.f32                              */
    GQ_PROBE_FFMA2 = 1,         /* fma.rn.f32x2                            */
    GQ_PROBE_FADD2 = 2,         /* add.rn.f32x2                            */
    GQ_PROBE_FADD = 3,          /* add.rn.f32                              */
    GQ_PROBE_DP4A = 4,          /* dp4a.u32.s32                            */
    GQ_PROBE_LOP3 = 5,          /* lop3.b32                                */
    GQ_PROBE_POPC = 6,          /* popc.b32                                */
    GQ_PROBE_PRMT = 7,          /* prmt.b32                                */
    GQ_PROBE_SHF = 8,           /* shf.l.wrap.b32                          */
    GQ_PROBE_IMAD = 9,          /* mad.lo.u32                              */
    GQ_PROBE_SHFL = 10,         /* shfl.sync.idx.b32                       */
    GQ_PROBE_LDS = 11,          /* ld.shared.u32, conflict-free (+ one lop3 each) */
    GQ_PROBE_DP4A_FFMA2 = 12,   /* dp4a and fma.rn.f32x2 interleaved       */
    GQ_PROBE_LDS_SHFL = 13,     /* ld.shared.u32 and shfl.sync interleaved */
    GQ_PROBE_FFMA_FFMA2 = 14,   /* fma.rn.f32 and fma.rn.f32x2 interleaved */
    GQ_PROBE_LOP3_DP4A = 15,    /* lop3 and dp4a interleaved               */
    GQ_PROBE_FADD_FFMA2 = 16,   /* add.rn.f32 and fma.rn.f32x2 interleaved */
    GQ_PROBE_LOP3_FFMA2 = 17,   /* lop3 and fma.rn.f32x2 interleaved       */
    GQ_PROBE_HMMA_F16 = 18,     /* mma.sync m16n8k16 f16 x f16 + f32 (4096 flop each)  */
    GQ_PROBE_HMMA_BF16 = 19,    /* mma.sync m16n8k16 bf16 x bf16 + f32 (4096 flop)     */
    GQ_PROBE_QMMA_E4M3 = 20,    /* mma.sync m16n8k32 e4m3 x e4m3 + f32 (8192 flop),
                                   operand conversion included                          */
    GQ_PROBE_IMMA_S8 = 21,      /* mma.sync m16n8k32 s8 x s8 + s32 (8192 op)           */
    GQ_PROBE_HMMA_MIX = 22,     /* f16 mma.sync : lop3 : lop3 : fma.rn.f32, 1:2:1      */
    GQ_PROBE_QMMA_MIX = 23,     /* e4m3 mma.sync : lop3 : lop3 : fma.rn.f32, 1:2:1     */
    GQ_PROBE_LOP3_POPC = 24,    /* lop3 and popc interleaved               */
    GQ_PROBE_ISSUE_KINDS = 25
};

/* Instruction issue rate: one block of 32 warps per SM runs `iters` loop iterations of 32
 * instructions of `kind` per thread on eight independent chains; cycles_device[sm] receives the
 * block's elapsed SM clock cycles (one u64 per SM, 8-byte aligned); sink_device is one u32 that
 * keeps the chains live.  Warp instructions per SM per cycle = gq_probe_issue_insts(kind, iters)
 * / cycles.  Errors: GQ_EINVAL_SHAPE for an unknown kind or iters outside [1, 2^24];
 * GQ_EINVAL_PTR; GQ_ECUDA. */
int gq_probe_issue(int kind, int iters, unsigned long long* cycles_device, uint32_t* sink_device,
                   gq_stream_t stream);
/* Warp instructions of the measured kind(s) that one block of gq_probe_issue executes. */
double gq_probe_issue_insts(int kind, int iters);

/* tcgen05 MMA kinds of gq_probe_mma.  There is no int8 kind: ptxas rejects tcgen05.mma
 * kind::i8 for sm_103a. */
enum gq_probe_mma_kind {
    GQ_PROBE_MMA_F16 = 0,       /* kind::f16, bf16 operands, f32 accumulator, K = 16 per MMA  */
    GQ_PROBE_MMA_F8 = 1,        /* kind::f8f6f4, e4m3 operands, f32 accumulator, K = 32       */
    GQ_PROBE_MMA_F16_TMEM_A = 2 /* kind::f16 as kind 0, with the A operand in tensor memory   */
};

/* tcgen05 MMA rate: on every SM one thread issues `iters` MMAs of M = 128, N = n, with both
 * operands in shared memory, into one TMEM accumulator, then waits (bounded) for them to
 * complete; cycles_device[sm] receives the SM clock cycles from the first issue to completion.
 * (Kind GQ_PROBE_MMA_F16_TMEM_A takes A from tensor memory, as the library's prefill does.)
 * Flops per MMA = 2 * 128 * n * K.  Errors: GQ_EUNSUPPORTED for another kind; GQ_EINVAL_SHAPE
 * unless n is a multiple of 16 in [16, 256] and 1 <= iters <= 100000; GQ_EINVAL_PTR; GQ_ECUDA. */
int gq_probe_mma(int kind, int n, int iters, unsigned long long* cycles_device, gq_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* GQ_H */
