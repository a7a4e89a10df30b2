// Q1_0 x Q8_0 arithmetic shared by the decode GEMVs and the GEMM: the activation-side constants of
// the dp4a lane sums and the fixed final reduction (the per-value steps; each kernel file builds
// its own launches around them).
//
// Arithmetic (browseml-gpu.js, header comment and Q1_DOT_WGSL / Q1_MM_WGSL / Q1_MM4_WGSL): per
// row, per block i of 128 weights (f16 d0 + 128 sign bits), per sub-block k of 32 weights
// (Q8_0 block 4i+k: f16 d1 + 32 int8) and lane l (weights 4l..4l+3):
//   s = sum(bit ? q : -q) with the negate wrapping as int8;  p = d1*s (exact);
//   ab[l] = p (k = 0) or ab[l] + p;  acc[l] = fma(d0, ab[l], acc[l]);
//   y = ((a0+a4)+(a2+a6)) + ((a1+a5)+(a3+a7)).
//
// How the integer lane sums are formed here (the same values, fewer instructions):
//  * -128 quants: a -128 term is -128 whatever the bit, so with q~ = q except -128 -> 0 and
//    C = sum q~ + 128*count(-128),  s = 2*D - C  where D = sum over set bits of q~.
//  * The repack stores each 32-bit sign word bit-transposed: packed bit 8c+l = weight 4l+c.
//    Then (w & (0x01010101 << l)) holds lane l's four bits, one per byte, each worth 2^l, and
//    a single dp4a against the activation word l (bytes q~_{4l..4l+3}) gives 2^l * D.
//  * The dp4a accumulator starts at bits(1.5*2^23) - (sigma/2)*C, so its result read as f32 is
//    exactly 1.5*2^23 + (sigma/2)*s (sigma = 2^max(l,1), the lane's mask weight; lane 0's bits
//    are shifted up by one).  Subtracting 1.5*2^23 is exact, and multiplying by d1*2/sigma
//    gives exactly d1*s, so ab = fma(d1*2/sigma, t, ab) is the pages' rounded add.
//  * Pairs of lanes run through the packed f32x2 add/mul/fma (two IEEE operations each).
#pragma once

#include "gq_internal.cuh"

namespace gq {
namespace {

constexpr int kRPT = 4;          // rows per lane in the GEMV (a warp covers one 128-row tile)
constexpr uint32_t kMagicBits = 0x4B400000u;   // 1.5 * 2^23: ulp 1 in [2^23, 2^24)
constexpr float kMagic = 12582912.0f;
constexpr int kConstWords = 24;  // per 32-activation sub-block: 8 quant words, 8 seeds, 8 scales

// Activation constants of one (sub-block, lane l) from its f16 d1 bits and its four quants
// (little-endian word): the quant word with -128 zeroed, the dp4a seed and d1 * 2/sigma.
__device__ __forceinline__ void lane_consts(uint32_t d1bits, uint32_t qw, int l, uint32_t& qt, uint32_t& seed,
                                            float& d1s) {
    const float d1 = f16_to_f32(d1bits);
    int C = 0;
    uint32_t t = 0;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int q = static_cast<int>(static_cast<int8_t>((qw >> (8 * c)) & 0xFFu));
        if (q == -128) {
            C += 128;
        } else {
            C += q;
            t |= (static_cast<uint32_t>(q) & 0xFFu) << (8 * c);
        }
    }
    const int half_sigma = (l <= 1) ? 1 : (1 << (l - 1));
    qt = t;
    seed = kMagicBits - static_cast<uint32_t>(half_sigma * C);
    d1s = __fmul_rn(d1, 1.0f / static_cast<float>(half_sigma));   // power of two: exact
}

// The same from a 34-byte Q8_0 block in memory (2-byte aligned).
__device__ __forceinline__ void act_lane_consts(const uint16_t* blk, int l, uint32_t& qt, uint32_t& seed,
                                                float& d1s) {
    lane_consts(blk[0], static_cast<uint32_t>(blk[1 + 2 * l]) | (static_cast<uint32_t>(blk[2 + 2 * l]) << 16), l,
                qt, seed, d1s);
}

// The same from f32 activations, quantized to Q8_0 on the way (the values gq_quantize_q8_0 would
// store): lane l of sub-block kg quantizes x[32 kg + 4 l .. + 3] (v, already loaded); the
// sub-block's eight lanes are eight consecutive, 8-aligned lanes of the warp, which exchange their
// amax.
__device__ __forceinline__ void lane_consts_f32(const float4 v, int l, uint32_t& qt, uint32_t& seed, float& d1s) {
    float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float dd = q8_0_scale(amax);
    const uint32_t qw = (static_cast<uint32_t>(q8_0_quant(v.x, amax, dd)) & 0xFFu) |
                        ((static_cast<uint32_t>(q8_0_quant(v.y, amax, dd)) & 0xFFu) << 8) |
                        ((static_cast<uint32_t>(q8_0_quant(v.z, amax, dd)) & 0xFFu) << 16) |
                        (static_cast<uint32_t>(q8_0_quant(v.w, amax, dd)) << 24);
    lane_consts(__half_as_ushort(__float2half_rn(dd)), qw, l, qt, seed, d1s);
}
__device__ __forceinline__ void act_lane_consts_f32(const float* x, int kg, int l, uint32_t& qt, uint32_t& seed,
                                                    float& d1s) {
    lane_consts_f32(*reinterpret_cast<const float4*>(x + static_cast<size_t>(kg) * 32 + 4 * l), l, qt, seed, d1s);
}

// The eight dp4a results of one 32-weight sub-block word (transposed layout) read as f32, i.e.
// 1.5 * 2^23 + (sigma_l/2) * s_l, as four pairs (lanes 0-1, 2-3, 4-5, 6-7).
__device__ __forceinline__ void lane_words(uint32_t w, const uint4& q0, const uint4& q1, const uint4& s0,
                                           const uint4& s1, float2 f[4]) {
    const int r0 = dp4a_us(__funnelshift_l(0u, w, 1) & 0x02020202u, q0.x, static_cast<int>(s0.x));   // SHF: ALU pipe
    const int r1 = dp4a_us(w & 0x02020202u, q0.y, static_cast<int>(s0.y));
    const int r2 = dp4a_us(w & 0x04040404u, q0.z, static_cast<int>(s0.z));
    const int r3 = dp4a_us(w & 0x08080808u, q0.w, static_cast<int>(s0.w));
    const int r4 = dp4a_us(w & 0x10101010u, q1.x, static_cast<int>(s1.x));
    const int r5 = dp4a_us(w & 0x20202020u, q1.y, static_cast<int>(s1.y));
    const int r6 = dp4a_us(w & 0x40404040u, q1.z, static_cast<int>(s1.z));
    const int r7 = dp4a_us(w & 0x80808080u, q1.w, static_cast<int>(s1.w));
    f[0] = make_float2(__int_as_float(r0), __int_as_float(r1));
    f[1] = make_float2(__int_as_float(r2), __int_as_float(r3));
    f[2] = make_float2(__int_as_float(r4), __int_as_float(r5));
    f[3] = make_float2(__int_as_float(r6), __int_as_float(r7));
}

// The eight lane values t_l = (sigma_l/2) * s_l (the words minus 1.5 * 2^23, exactly).
__device__ __forceinline__ void lane_values(uint32_t w, const uint4& q0, const uint4& q1, const uint4& s0,
                                            const uint4& s1, float2 t[4]) {
    lane_words(w, q0, q1, s0, s1, t);
    const float2 nm = make_float2(-kMagic, -kMagic);
#pragma unroll
    for (int p = 0; p < 4; ++p) t[p] = fadd2(t[p], nm);
}

__device__ __forceinline__ float final_reduce(const float2 acc[4]) {
    // acc[0] = (a0,a1), acc[1] = (a2,a3), acc[2] = (a4,a5), acc[3] = (a6,a7)
    const float2 s0415 = fadd2(acc[0], acc[2]);     // (a0+a4, a1+a5)
    const float2 s2637 = fadd2(acc[1], acc[3]);     // (a2+a6, a3+a7)
    const float2 lohi = fadd2(s0415, s2637);        // ((a0+a4)+(a2+a6), (a1+a5)+(a3+a7))
    return __fadd_rn(lohi.x, lohi.y);
}

}  // namespace
}  // namespace gq
