// The C ABI of libgq: argument validation on the host, then one launch on the caller's stream.
// Nothing here allocates device memory or synchronizes, except gq_device_error().
#include <algorithm>
#include <cstdint>

#include "gq_internal.cuh"
#include "wq_mma.cuh"
#include "w1a32_mma.cuh"

namespace {

thread_local int t_last_cuda_error = 0;

constexpr int kMaxK = 65536;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return GQ_OK;
    t_last_cuda_error = static_cast<int>(e);
    return GQ_ECUDA;
}

int check_q1(const void* packed, const void* act, const float* y, int rows, int n) {
    if (rows < 1 || n < 128 || n % 128 != 0 || n > gq::kMaxN) return GQ_EINVAL_SHAPE;
    if (!packed || !act || !y) return GQ_EINVAL_PTR;
    if (!aligned(packed, 16) || !aligned(act, 2) || !aligned(y, 4)) return GQ_EINVAL_PTR;
    return GQ_OK;
}

}  // namespace

namespace gq {
void record_cuda_error(int err) { t_last_cuda_error = err; }
}  // namespace gq

extern "C" {

const char* gq_version(void) { return "gq 0.1.0 (sm_103a)"; }

const char* gq_status_string(int status) {
    switch (status) {
        case GQ_OK: return "ok";
        case GQ_EINVAL_SHAPE: return "invalid shape";
        case GQ_EINVAL_PTR: return "invalid pointer (null or misaligned)";
        case GQ_EUNSUPPORTED: return "unsupported path";
        case GQ_ECUDA: return "CUDA launch error";
        default: return "unknown status";
    }
}

int gq_last_cuda_error(void) { return t_last_cuda_error; }

int gq_device_error(void) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_status(e) == GQ_OK ? 0 : -1;
    const unsigned v = gq::error_read_clear_q1() | gq::error_read_clear_q1_gemv() | gq::error_read_clear_ternary() | gq::error_read_clear_prefill_mma() |
                       gq::error_read_clear_wq_mma() | gq::error_read_clear_w1a32() | gq::error_read_clear_probes() |
                       gq::error_read_clear_block_q8();
    return v == ~0u ? -1 : static_cast<int>(v);
}

size_t gq_q1_0_packed_bytes(int rows, int n) {
    if (rows < 1 || n < 128 || n % 128 != 0 || n > gq::kMaxN) return 0;
    const size_t tiles = (static_cast<size_t>(rows) + gq::kTileRows - 1) / gq::kTileRows;
    return tiles * static_cast<size_t>(n / 128) * gq::kChunkBytes;
}

int gq_q1_0_pack(const void* raw, int rows, int n, void* packed, gq_stream_t stream) {
    if (rows < 1 || n < 128 || n % 128 != 0 || n > gq::kMaxN) return GQ_EINVAL_SHAPE;
    if (!raw || !packed || !aligned(packed, 16)) return GQ_EINVAL_PTR;
    return cuda_status(gq::launch_q1_pack(raw, rows, n, packed, reinterpret_cast<cudaStream_t>(stream)));
}

size_t gq_q1_q8_workspace_bytes(int n) {
    if (n < 128 || n % 128 != 0 || n > gq::kMaxN) return 0;
    return gq::gemv_workspace_bytes(n);
}

int q1_q8_gemv(const void* packed_w, const void* act, float* y, int rows, int n, void* workspace,
               gq_stream_t stream) {
    const int st = check_q1(packed_w, act, y, rows, n);
    if (st != GQ_OK) return st;
    if (!workspace || !aligned(workspace, 16)) return GQ_EINVAL_PTR;
    return cuda_status(gq::launch_q1_gemv(packed_w, act, y, rows, n, workspace, GQ_ACT_Q8_0,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

int q1_q8_gemv_raw(const void* w_q1_0, const void* act, float* y, int rows, int n, gq_stream_t stream) {
    if (rows < 1 || n < 128 || n % 128 != 0 || n > gq::kMaxN) return GQ_EINVAL_SHAPE;
    if (!w_q1_0 || !act || !y || !aligned(w_q1_0, 2) || !aligned(act, 2) || !aligned(y, 4)) return GQ_EINVAL_PTR;
    return cuda_status(gq::launch_q1_gemv_raw(w_q1_0, act, y, rows, n, reinterpret_cast<cudaStream_t>(stream)));
}

int gq_pack_q8_0(const void* raw_q8_0, int cols, int n, float* d, uint32_t* q, gq_stream_t stream) {
    if (cols < 1 || n < 32 || n % 32 != 0 || n > gq::kMaxN) return GQ_EINVAL_SHAPE;
    if (!raw_q8_0 || !d || !q || !aligned(raw_q8_0, 2) || !aligned(d, 4) || !aligned(q, 4)) return GQ_EINVAL_PTR;
    return cuda_status(gq::launch_pack_q8_0(raw_q8_0, cols, n, d, q, reinterpret_cast<cudaStream_t>(stream)));
}

int q1_q8_gemv_f32(const void* packed_w, const float* x, float* y, int rows, int n, void* workspace,
                   gq_stream_t stream) {
    const int st = check_q1(packed_w, x, y, rows, n);
    if (st != GQ_OK) return st;
    if (!aligned(x, 16) || !workspace || !aligned(workspace, 16)) return GQ_EINVAL_PTR;
    return cuda_status(gq::launch_q1_gemv(packed_w, x, y, rows, n, workspace, GQ_ACT_F32,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

int gq_gemv_group_plan(gq_gemv_desc* descs, int count, int* total_tiles) {
    if (!descs || !total_tiles) return GQ_EINVAL_PTR;
    if (count < 1 || count > 65535) return GQ_EINVAL_SHAPE;
    for (int i = 0; i < count; ++i) {
        const int st = check_q1(descs[i].packed_w, descs[i].act, descs[i].y, descs[i].rows, descs[i].n);
        if (st != GQ_OK) return st;
        if (descs[i].act_format != GQ_ACT_Q8_0 && descs[i].act_format != GQ_ACT_F32) return GQ_EINVAL_SHAPE;
        if (descs[i].act_format == GQ_ACT_F32 && !aligned(descs[i].act, 16)) return GQ_EINVAL_PTR;
        if (!descs[i].workspace || !aligned(descs[i].workspace, 16)) return GQ_EINVAL_PTR;
    }
    // Largest n first (stable): the kernel hands tiles to warps in snake order over this list.
    std::stable_sort(descs, descs + count,
                     [](const gq_gemv_desc& a, const gq_gemv_desc& b) { return a.n > b.n; });
    long long tiles = 0;
    for (int i = 0; i < count; ++i) {
        descs[i].tile_begin = static_cast<int>(tiles);
        tiles += gq::gemv_tiles_for(descs[i].rows);
        if (tiles > 0x7fffffffLL) return GQ_EINVAL_SHAPE;
    }
    *total_tiles = static_cast<int>(tiles);
    return GQ_OK;
}

int q1_q8_gemv_grouped(const gq_gemv_desc* descs, int count, int total_tiles, int* counter, gq_stream_t stream) {
    if (!descs || !aligned(descs, 8) || !counter || !aligned(counter, 4)) return GQ_EINVAL_PTR;
    if (count < 1 || count > 65535 || total_tiles < 1) return GQ_EINVAL_SHAPE;
    return cuda_status(
        gq::launch_q1_gemv_grouped(descs, count, total_tiles, counter, reinterpret_cast<cudaStream_t>(stream)));
}

int q1_q8_gemm(const void* packed_w, const void* act, float* y, int rows, int n, int cols, int path,
               gq_stream_t stream) {
    const int st = check_q1(packed_w, act, y, rows, n);
    if (st != GQ_OK) return st;
    if (cols < 1 || cols > 65535 * 4) return GQ_EINVAL_SHAPE;
    if (path == GQ_PATH_AUTO) path = GQ_PATH_DP4A;
    if (path != GQ_PATH_DP4A && path != GQ_PATH_LUT4) return GQ_EUNSUPPORTED;
    return cuda_status(gq::launch_q1_gemm(packed_w, act, y, rows, n, cols, path, reinterpret_cast<cudaStream_t>(stream)));
}

int block_q8_matmul_nt(const float* x, const uint32_t* quants, const float* scales, float* y, int m, int k, int n,
                       gq_stream_t stream) {
    if (m < 1 || k < 32 || n < 1 || k % 32 != 0 || k > kMaxK || m > 65535 * 16) return GQ_EINVAL_SHAPE;
    if (!x || !quants || !scales || !y) return GQ_EINVAL_PTR;
    if (!aligned(x, 4) || !aligned(quants, 16) || !aligned(scales, 4) || !aligned(y, 4)) return GQ_EINVAL_PTR;
    return cuda_status(gq::launch_block_q8(x, quants, scales, y, m, k, n, reinterpret_cast<cudaStream_t>(stream)));
}

int q1s32_f32_gemm(const uint32_t* signs, const float* wscale, const float* x, float* y, int M, int N, int K, int path,
                   gq_stream_t stream) {
    if (N < 1 || M < 1 || M > 65535 || K < 32 || K % 32 != 0 || K > kMaxK) return GQ_EINVAL_SHAPE;
    if (path == GQ_PATH_AUTO) path = GQ_PATH_LUT4;
    if (path != GQ_PATH_LUT4 && path != GQ_PATH_FMA) return GQ_EUNSUPPORTED;
    if (!signs || !wscale || !x || !y) return GQ_EINVAL_PTR;
    if (!aligned(signs, 4) || !aligned(wscale, 4) || !aligned(x, 16) || !aligned(y, 4)) return GQ_EINVAL_PTR;
    return cuda_status(
        gq::launch_q1s32_f32(signs, wscale, x, y, M, N, K, path, reinterpret_cast<cudaStream_t>(stream)));
}

size_t gq_q1s32_mma_workspace_bytes(int M, int K) {
    if (M < 1 || M > 65535 * 128 || K < 64 || K % 64 != 0 || K > kMaxK) return 0;
    return gq::w1a32_mma_workspace_bytes(M, K);
}

int q1s32_f32_gemm_mma(const uint32_t* signs, const float* wscale, const float* x, float* y, int M, int N, int K,
                       void* workspace, gq_stream_t stream) {
    if (N < 1 || M < 1 || M > 65535 * 128 || K < 64 || K % 64 != 0 || K > kMaxK) return GQ_EINVAL_SHAPE;
    if (!signs || !wscale || !x || !y || !workspace) return GQ_EINVAL_PTR;
    if (!aligned(signs, 16) || !aligned(wscale, 8) || !aligned(x, 4) || !aligned(y, 4) || !aligned(workspace, 16))
        return GQ_EINVAL_PTR;
    return cuda_status(
        gq::launch_w1a32_mma(signs, wscale, x, y, M, N, K, workspace, reinterpret_cast<cudaStream_t>(stream)));
}

static int wq_call(int bits, const uint32_t* w, const float* scale, const float* x, float* y, int T, int N, int K,
                   gq_stream_t stream) {
    if (N < 1 || T < 1 || T > 65535 * 128 || K < 32 || K % 32 != 0 || K > kMaxK) return GQ_EINVAL_SHAPE;
    if (!w || !scale || !x || !y) return GQ_EINVAL_PTR;
    if (!aligned(w, 16) || !aligned(scale, 4) || !aligned(x, 16) || !aligned(y, 4)) return GQ_EINVAL_PTR;
    return cuda_status(gq::launch_wq(bits, w, scale, x, y, T, N, K, reinterpret_cast<cudaStream_t>(stream)));
}

int matvec_q8(const uint32_t* w, const float* scale, const float* x, float* y, int N, int K, gq_stream_t stream) {
    return wq_call(8, w, scale, x, y, 1, N, K, stream);
}
int matmul_q8(const uint32_t* w, const float* scale, const float* x, float* y, int T, int N, int K,
              gq_stream_t stream) {
    return wq_call(8, w, scale, x, y, T, N, K, stream);
}
size_t gq_wq_mma_workspace_bytes(int T, int K) {
    if (T < 1 || T > 65535 * 128 || K < 64 || K % 32 != 0 || K > kMaxK) return 0;
    return gq::wq_mma_workspace_bytes(T, K);
}

static int wq_mma_call(int bits, const uint32_t* w, const float* scale, const float* x, float* y, int T, int N, int K,
                       void* workspace, gq_stream_t stream) {
    if (N < 1 || T < 1 || T > 65535 * 128 || K < 64 || K % 32 != 0 || K > kMaxK) return GQ_EINVAL_SHAPE;
    if (!w || !scale || !x || !y || !workspace) return GQ_EINVAL_PTR;
    if (!aligned(w, 16) || !aligned(scale, 4) || !aligned(x, 16) || !aligned(y, 4) || !aligned(workspace, 16))
        return GQ_EINVAL_PTR;
    return cuda_status(
        gq::launch_wq_mma(bits, w, scale, x, y, T, N, K, workspace, reinterpret_cast<cudaStream_t>(stream)));
}

int matmul_q8_mma(const uint32_t* w, const float* scale, const float* x, float* y, int T, int N, int K,
                  void* workspace, gq_stream_t stream) {
    return wq_mma_call(8, w, scale, x, y, T, N, K, workspace, stream);
}
int matmul_q4g128_mma(const uint32_t* w, const float* scale, const float* x, float* y, int T, int N, int K,
                      void* workspace, gq_stream_t stream) {
    return wq_mma_call(4, w, scale, x, y, T, N, K, workspace, stream);
}

int matvec_q4g128(const uint32_t* w, const float* scale, const float* x, float* y, int N, int K, gq_stream_t stream) {
    return wq_call(4, w, scale, x, y, 1, N, K, stream);
}
int matmul_q4g128(const uint32_t* w, const float* scale, const float* x, float* y, int T, int N, int K,
                  gq_stream_t stream) {
    return wq_call(4, w, scale, x, y, T, N, K, stream);
}

int ternary_bitplane_gemv(const uint32_t* P, const uint32_t* N, const uint32_t* X, int32_t* y, int rows, int k,
                          int batch, gq_stream_t stream) {
    if (rows < 1 || k < 1024 || batch < 1 || k % 1024 != 0 || k > kMaxK || batch > 64) return GQ_EINVAL_SHAPE;
    if (!P || !N || !X || !y) return GQ_EINVAL_PTR;
    if (!aligned(P, 16) || !aligned(N, 16) || !aligned(X, 16) || !aligned(y, 4)) return GQ_EINVAL_PTR;
    return cuda_status(gq::launch_ternary(P, N, X, y, rows, k, batch, reinterpret_cast<cudaStream_t>(stream)));
}

int gq_quantize_q8_0(const float* x, int m, int k, uint16_t* d, int8_t* q, uint16_t* op, gq_stream_t stream) {
    if (m < 1 || k < 32 || k % 32 != 0 || k > kMaxK) return GQ_EINVAL_SHAPE;
    if (!x || !d || !q) return GQ_EINVAL_PTR;
    if (!aligned(x, 4) || !aligned(d, 2) || !aligned(q, 16) || (op && !aligned(op, 16))) return GQ_EINVAL_PTR;
    return cuda_status(gq::launch_quantize(x, m, k, d, q, op, reinterpret_cast<cudaStream_t>(stream)));
}

int q1s32_q8_gemm(const uint32_t* signs, const float* wscale, const uint16_t* xd, const int8_t* xq,
                  const uint16_t* xq_mma, float* y, int M, int N, int K, int path, gq_stream_t stream) {
    if (M < 1 || N < 1 || K < 64 || K % 64 != 0 || K > kMaxK || M > 65535 * 32) return GQ_EINVAL_SHAPE;
    if (path == GQ_PATH_AUTO) path = (xq_mma && M >= 64) ? GQ_PATH_MMA : GQ_PATH_LUT4;
    if (path != GQ_PATH_LUT4 && path != GQ_PATH_MMA) return GQ_EUNSUPPORTED;
    if (!signs || !wscale || !xd || !xq || !y) return GQ_EINVAL_PTR;
    if (!aligned(signs, 16) || !aligned(wscale, 4) || !aligned(xd, 4) || !aligned(xq, 16) || !aligned(y, 4))
        return GQ_EINVAL_PTR;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (path == GQ_PATH_MMA) {
        if (!xq_mma || !aligned(xq_mma, 16) || !aligned(wscale, 8)) return GQ_EINVAL_PTR;   // row scales as pairs
        const cudaError_t e = gq::launch_prefill_mma(signs, wscale, xd, xq_mma, y, M, N, K, s);
        if (e == cudaErrorNotSupported) return GQ_EUNSUPPORTED;
        return cuda_status(e);
    }
    return cuda_status(gq::launch_prefill_lut4(signs, wscale, xd, xq, y, M, N, K, s));
}

}  // extern "C"
