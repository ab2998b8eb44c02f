// quantize.cu -- MX microscaling of bf16 tensors (32-element blocks, one
// shared E8M0 scale each) for MXFP8 (E4M3), MXFP6 (E2M3) and MXFP4 (E2M1).
//
// Method: "Fused-Softmax shifts an AI attention bottleneck onto faster GPU
// hardware", paragraphs 7-8 (MX operands of the three formats) and
// "EFQ-Softmax: Exp-Free Quantization for Softmax", section "B. Block-Scaled
// E2M1 Probability Representation" (exponent-only block scale).  The scale
// rule -- the smallest power of two 2^X with amax <= max_elem * 2^X -- is
// this library's reading; the pages print none.
//
// Both kernels stream their input once and write codes + scales once: they
// are HBM-bound, so the design goal is full-sector, coalesced traffic.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fsa_internal.h"
#include "sm100_ptx.cuh"

namespace fsa {
namespace {

struct FmtConsts {
    int emax;       // exponent of the largest finite element
    uint32_t mthr;  // largest element = (1 + mthr / 128) * 2^emax in bf16 mantissa units
};

__device__ __forceinline__ FmtConsts fmt_consts(int elem) {
    if (elem == ELEM_E4M3) return {8, 0x60};  // 448 = 1.75 * 2^8
    if (elem == ELEM_E2M3) return {2, 0x70};  // 7.5 = 1.875 * 2^2
    return {2, 0x40};                         // 6   = 1.5 * 2^2
}

// Smallest integer X with amax <= max_elem * 2^X, clamped to [-127, 127];
// -127 for an all-zero block.  amax is given as the bit pattern of a
// non-negative bf16 (its magnitude bits, 15 bits).
__device__ __forceinline__ int mx_scale_exp(uint32_t amax_bf16, FmtConsts f) {
    if (amax_bf16 == 0) return -127;
    int E = static_cast<int>(amax_bf16 >> 7);
    uint32_t m = amax_bf16 & 0x7Fu;
    int e;
    if (E == 0) {  // bf16 subnormal: m * 2^-133, renormalise
        int nb = 32 - __clz(m);
        e = nb - 134;
        m = (m << (8 - nb)) & 0x7Fu;
    } else {
        e = E - 127;
    }
    int X = e - f.emax + (m > f.mthr ? 1 : 0);
    return min(127, max(-127, X));
}

// 2^-X as an FP32 (X in [-127, 126] for any bf16 block maximum).
__device__ __forceinline__ float pow2_neg(int X) {
    return __int_as_float((127 - X) << 23);
}

// Codes of two scaled values: byte 0 = code(lo), byte 1 = code(hi).
__device__ __forceinline__ uint32_t encode_pair(int elem, float lo, float hi) {
    if (elem == ELEM_E4M3) return cvt_e4m3x2(lo, hi);
    if (elem == ELEM_E2M3) return cvt_e2m3x2(lo, hi);
    uint32_t n = cvt_e2m1x2(lo, hi);
    return (n & 0xFu) | ((n >> 4) << 8);
}

// Value of a narrow code (E2M3 or E2M1), exactly.
__device__ __forceinline__ float decode_narrow(int elem, uint32_t c) {
    uint32_t s, e, m;
    float mag;
    if (elem == ELEM_E2M3) {
        s = (c >> 5) & 1u; e = (c >> 3) & 3u; m = c & 7u;
        mag = e ? static_cast<float>(8u + m) * __int_as_float((127 + static_cast<int>(e) - 4) << 23)
                : static_cast<float>(m) * 0.125f;
    } else {
        s = (c >> 3) & 1u; e = (c >> 1) & 3u; m = c & 1u;
        mag = e ? static_cast<float>(2u + m) * __int_as_float((127 + static_cast<int>(e) - 2) << 23)
                : static_cast<float>(m) * 0.5f;
    }
    return s ? -mag : mag;
}

// Pair of element codes -> pair of E4M3 bit patterns of the same values.
__device__ __forceinline__ uint32_t to_e4m3_container(int elem, uint32_t pair) {
    if (elem == ELEM_E4M3) return pair;
    return cvt_e4m3x2(decode_narrow(elem, pair & 0xFFu), decode_narrow(elem, (pair >> 8) & 0xFFu));
}

// Quantizes 32 values v[] (n valid, rest zero) held as bf16 bit patterns.
// Writes 8 words of packed codes (4 per word, element i in byte i % 4 of
// word i / 4) and returns X.
__device__ __forceinline__ int quantize_block32(const uint32_t (&h)[32], int elem, int layout,
                                                uint32_t (&w)[8]) {
    uint32_t amax = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = max(amax, h[i] & 0x7FFFu);
    const int X = mx_scale_exp(amax, fmt_consts(elem));
    const float sc = pow2_neg(X);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float a = __uint_as_float(h[4 * i + 0] << 16) * sc;
        float b = __uint_as_float(h[4 * i + 1] << 16) * sc;
        float c = __uint_as_float(h[4 * i + 2] << 16) * sc;
        float d = __uint_as_float(h[4 * i + 3] << 16) * sc;
        uint32_t p0 = encode_pair(elem, a, b), p1 = encode_pair(elem, c, d);
        if (layout == QL_ATTN) {
            p0 = to_e4m3_container(elem, p0);
            p1 = to_e4m3_container(elem, p1);
        }
        w[i] = (p0 & 0xFFFFu) | (p1 << 16);
    }
    return X;
}

// 2^X as an FP32 for X in [-127, 127] (2^-127 is subnormal).
__device__ __forceinline__ float pow2f(int X) {
    return X >= -126 ? __int_as_float((127 + X) << 23) : __int_as_float(0x00400000);
}

// Sum of squares of the 32 values of one quantized block: the E4M3 patterns
// in w (ATTN layout) decoded exactly (E4M3 -> f16 is exact), times 4^X.
// Overflows to +inf for huge blocks; a block below 2^-60 may round to zero,
// which the absolute slack of the row bound covers.
__device__ __forceinline__ float block_sumsq(const uint32_t (&w)[8], int X) {
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t f16x2;
            asm("{\n.reg .b16 t;\ncvt.u16.u32 t, %1;\ncvt.rn.f16x2.e4m3x2 %0, t;\n}"
                : "=r"(f16x2) : "r"(w[i] >> (16 * h)));
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&f16x2));
            s = __fmaf_rn(f.x, f.x, s);
            s = __fmaf_rn(f.y, f.y, s);
        }
    }
    const float p = pow2f(X);
    return s * p * p;
}

// Upper bound of a row's Euclidean norm from the FP32 sum of its squares:
// the relative slack covers the rounding of the 128 squares' sum and of the
// square root, the absolute one blocks that underflowed.
__device__ __forceinline__ float norm_bound(float sumsq) {
    return __fmaf_rn(sqrtf(sumsq), 1.0f + 1.0f / 1024.0f, 1e-18f);
}

__device__ __forceinline__ int atom_offset(int64_t r_in_tile, int kb) {
    return static_cast<int>((r_in_tile & 31) * 16 + (r_in_tile >> 5) * 4 + kb);
}

// Blocks of 32 along the last axis.  One thread per block.
__global__ void quant_rows_kernel(const uint16_t* __restrict__ x, int64_t lines, int64_t cols,
                                  int elem, int layout, uint8_t* __restrict__ codes,
                                  uint8_t* __restrict__ scales, int64_t rows_per_mat, int vec,
                                  float* __restrict__ norms, int norm_mode) {
    const int64_t nblk = (cols + 31) / 32;
    const int64_t total = lines * nblk;
    const int64_t n_tiles = (rows_per_mat + kTile - 1) / kTile;
    for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t line = idx / nblk;
        const int kb = static_cast<int>(idx - line * nblk);
        const int64_t c0 = static_cast<int64_t>(kb) * 32;
        const int n = static_cast<int>(cols - c0 < 32 ? cols - c0 : 32);
        const uint16_t* src = x + line * cols + c0;
        uint32_t h[32];
        if (vec && n == 32) {
            const uint4* s4 = reinterpret_cast<const uint4*>(src);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint4 u = __ldg(s4 + i);
                h[8 * i + 0] = u.x & 0xFFFFu; h[8 * i + 1] = u.x >> 16;
                h[8 * i + 2] = u.y & 0xFFFFu; h[8 * i + 3] = u.y >> 16;
                h[8 * i + 4] = u.z & 0xFFFFu; h[8 * i + 5] = u.z >> 16;
                h[8 * i + 6] = u.w & 0xFFFFu; h[8 * i + 7] = u.w >> 16;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) h[i] = i < n ? static_cast<uint32_t>(__ldg(src + i)) : 0u;
        }
        uint32_t w[8];
        const int X = quantize_block32(h, elem, layout, w);
        uint8_t* dst = codes + line * cols + c0;
        if (vec && n == 32 && (cols % 16) == 0) {
            uint4* d4 = reinterpret_cast<uint4*>(dst);
            d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
            d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
        } else {
            for (int i = 0; i < n; ++i) dst[i] = static_cast<uint8_t>(w[i >> 2] >> (8 * (i & 3)));
        }
        const uint8_t sb = static_cast<uint8_t>(X + 127);
        if (layout == QL_PLAIN) {
            scales[line * nblk + kb] = sb;
        } else {
            const int64_t mat = line / rows_per_mat, r = line - mat * rows_per_mat;
            scales[(mat * n_tiles + r / kTile) * kAtomBytes + atom_offset(r % kTile, kb)] = sb;
            if (norm_mode != NORM_NONE) {
                // the nblk blocks of a row sit in nblk consecutive lanes: the
                // warp's indices are consecutive, nblk divides 32 and total is
                // a multiple of nblk, so a row's lanes are active together;
                // the lanes of this pass are those below total
                const int64_t base = idx - (threadIdx.x & 31);
                const int64_t left = total - base;
                const unsigned act = left >= 32 ? 0xFFFFFFFFu : (1u << left) - 1u;
                float ss = block_sumsq(w, X);
                for (int o = 1; o < nblk; o <<= 1) ss += __shfl_xor_sync(act, ss, o);
                if (kb == 0) {
                    const float bnd = norm_bound(ss);
                    if (norm_mode == NORM_ROW)
                        norms[line] = bnd;
                    else  // non-negative floats order like their bit patterns
                        atomicMax(reinterpret_cast<unsigned int*>(norms + mat * n_tiles + r / kTile),
                                  __float_as_uint(bnd));
                }
            }
        }
    }
}

// Blocks of 32 along the middle axis (rows); output transposed so that each
// block becomes 32 contiguous code bytes of line `col`.  A CTA stages a
// 32-row x 128-column tile in shared memory with coalesced loads.
constexpr int kColTileC = 128;
__global__ void __launch_bounds__(256) quant_cols_kernel(const uint16_t* __restrict__ x,
                                                         int64_t rows, int64_t cols, int elem,
                                                         int layout, uint8_t* __restrict__ codes,
                                                         int64_t pitch,
                                                         uint8_t* __restrict__ scales) {
    __shared__ uint16_t tile[32][kColTileC + 2];
    const int64_t b = blockIdx.z;
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * 32;
    const int64_t c0 = static_cast<int64_t>(blockIdx.y) * kColTileC;
    const uint16_t* xb = x + b * rows * cols;
    for (int i = threadIdx.x; i < 32 * kColTileC; i += blockDim.x) {
        const int rr = i / kColTileC, cc = i % kColTileC;
        const int64_t r = r0 + rr, c = c0 + cc;
        tile[rr][cc] = (r < rows && c < cols) ? __ldg(xb + r * cols + c) : static_cast<uint16_t>(0);
    }
    __syncthreads();
    const int cc = threadIdx.x;
    const int64_t c = c0 + cc;
    if (cc >= kColTileC || c >= cols) return;
    uint32_t h[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) h[i] = tile[i][cc];
    uint32_t w[8];
    const int X = quantize_block32(h, elem, layout, w);
    const int64_t nblk = (rows + 31) / 32;
    const int kb = static_cast<int>(r0 / 32);
    const uint8_t sb = static_cast<uint8_t>(X + 127);
    uint8_t* dst = codes + (b * cols + c) * pitch + r0;
    if (layout == QL_PLAIN) {
        const int n = static_cast<int>(rows - r0 < 32 ? rows - r0 : 32);
        for (int i = 0; i < n; ++i) dst[i] = static_cast<uint8_t>(w[i >> 2] >> (8 * (i & 3)));
        scales[(b * cols + c) * nblk + kb] = sb;
    } else {
        // pitch is a multiple of 16 and r0 of 32: each 16-byte half of the
        // block is entirely inside or entirely outside the padded line; the
        // padding keys [rows, pitch) receive zero codes (loaded as zeros).
        uint4* d4 = reinterpret_cast<uint4*>(dst);
        d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
        if (r0 + 16 < pitch) d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
        const int64_t n_tiles = (rows + kTile - 1) / kTile;
        scales[(b * n_tiles + r0 / kTile) * kAtomBytes + atom_offset(c, kb & 3)] = sb;
    }
}


// ---------------------------------------------------------------------------
// Attention layout (E4M3 containers, scale atoms), the fused attention's
// operands.  Specialised per element type; a row of D = 64 or 128 values has
// nblk = 2 or 4 blocks, one thread per block, so every index is a shift or a
// 32-bit division once per block.

// Largest magnitude of 32 bf16 values held as 16 packed pairs (sign bits off,
// then a 16-bit two-way max: magnitudes order like their bit patterns).
__device__ __forceinline__ uint32_t amax_pairs(const uint32_t (&u)[16]) {
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint32_t a = u[i] & 0x7FFF7FFFu;
        asm("max.u16x2 %0, %0, %1;" : "+r"(m) : "r"(a));
    }
    return max(m & 0xFFFFu, m >> 16);
}

// bf16 pair -> two FP32 values scaled by sc (exact: sc is a power of two and
// no bf16 block element drops below the FP32 normal range after scaling).
__device__ __forceinline__ float2 scale_pair(uint32_t u, float2 sc) {
    return __fmul2_rn(make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u)), sc);
}

// E4M3 bytes of four E2M1 values: E2M1 -> f16 -> E4M3 are exact conversions.
__device__ __forceinline__ uint32_t e2m1x4_as_e4m3(float a0, float a1, float a2, float a3) {
    uint32_t r;
    asm("{\n.reg .b8 n0, n1;\n.reg .b32 h0, h1;\n.reg .b16 e0, e1;\n"
        "cvt.rn.satfinite.e2m1x2.f32 n0, %2, %1;\n"
        "cvt.rn.satfinite.e2m1x2.f32 n1, %4, %3;\n"
        "cvt.rn.f16x2.e2m1x2 h0, n0;\n"
        "cvt.rn.f16x2.e2m1x2 h1, n1;\n"
        "cvt.rn.satfinite.e4m3x2.f16x2 e0, h0;\n"
        "cvt.rn.satfinite.e4m3x2.f16x2 e1, h1;\n"
        "mov.b32 %0, {e0, e1};\n}"
        : "=r"(r) : "f"(a0), "f"(a1), "f"(a2), "f"(a3));
    return r;
}

// Sum of squares of four E4M3 bytes (exact decode to f16, FP32 accumulation).
__device__ __forceinline__ float sumsq_e4m3x4(uint32_t w, float s) {
    asm("{\n.reg .b16 p0, p1, a, b, c, d;\n.reg .b32 h0, h1;\n"
        "mov.b32 {p0, p1}, %1;\n"
        "cvt.rn.f16x2.e4m3x2 h0, p0;\n"
        "cvt.rn.f16x2.e4m3x2 h1, p1;\n"
        "mov.b32 {a, b}, h0;\n"
        "mov.b32 {c, d}, h1;\n"
        "fma.rn.f32.f16 %0, a, a, %0;\n"
        "fma.rn.f32.f16 %0, b, b, %0;\n"
        "fma.rn.f32.f16 %0, c, c, %0;\n"
        "fma.rn.f32.f16 %0, d, d, %0;\n}"
        : "+f"(s) : "r"(w));
    return s;
}

// Quantizes one block of 32 bf16 values (16 pairs) into 8 words of E4M3
// containers; returns the stored scale exponent.  E2M3 values v are stored
// as the E4M3 pattern of v / 64 with exponent X + 6: rounding to E4M3 there
// is rounding to E2M3 (the same three mantissa bits, E2M3's subnormal step
// 1/8 is E4M3's 2^-9 shifted by 2^6), and the products are unchanged.
template <int kElem>
__device__ __forceinline__ int quantize_block_attn(const uint32_t (&u)[16], uint32_t (&w)[8]) {
    constexpr FmtConsts f = kElem == ELEM_E4M3 ? FmtConsts{8, 0x60}
                                               : (kElem == ELEM_E2M3 ? FmtConsts{2, 0x70} : FmtConsts{2, 0x40});
    int X = mx_scale_exp(amax_pairs(u), f);
    if (kElem == ELEM_E2M3 && X <= 121) {
        const float sc = pow2_neg(X + 6);
        const float2 s2 = make_float2(sc, sc);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float2 a = scale_pair(u[2 * i], s2), b = scale_pair(u[2 * i + 1], s2);
            w[i] = cvt_e4m3x4(a.x, a.y, b.x, b.y);
        }
        return X + 6;
    }
    const float sc = pow2_neg(X);
    const float2 s2 = make_float2(sc, sc);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float2 a = scale_pair(u[2 * i], s2), b = scale_pair(u[2 * i + 1], s2);
        if (kElem == ELEM_E4M3) {
            w[i] = cvt_e4m3x4(a.x, a.y, b.x, b.y);
        } else if (kElem == ELEM_E2M1) {
            w[i] = e2m1x4_as_e4m3(a.x, a.y, b.x, b.y);
        } else {  // E2M3 block with X > 121 (magnitudes near the bf16 maximum)
            const uint32_t p0 = to_e4m3_container(ELEM_E2M3, cvt_e2m3x2(a.x, a.y));
            const uint32_t p1 = to_e4m3_container(ELEM_E2M3, cvt_e2m3x2(b.x, b.y));
            w[i] = (p0 & 0xFFFFu) | (p1 << 16);
        }
    }
    return X;
}

// Q and K: lines of D = 64 or 128 bf16 values (lines = B*H*rows), blocks
// along D.  Optional row-norm bounds (NORM_ROW / NORM_TILE_MAX).
template <int kElem>
__global__ void __launch_bounds__(256) quant_rows_attn_kernel(
    const uint4* __restrict__ x, int lines, int log2_nblk, int rows_per_mat, uint4* __restrict__ codes,
    uint8_t* __restrict__ scales, float* __restrict__ norms, int norm_mode) {
    const int nblk = 1 << log2_nblk;
    const int total = lines << log2_nblk;
    const int n_tiles = (rows_per_mat + kTile - 1) / kTile;
    for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += gridDim.x * blockDim.x) {
        // a block is 64 bytes of input and 32 of output: uint4 units 4 and 2
        uint32_t u[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 v = __ldg(x + 4 * static_cast<int64_t>(idx) + i);
            u[4 * i] = v.x; u[4 * i + 1] = v.y; u[4 * i + 2] = v.z; u[4 * i + 3] = v.w;
        }
        uint32_t w[8];
        const int X = quantize_block_attn<kElem>(u, w);
        codes[2 * static_cast<int64_t>(idx)] = make_uint4(w[0], w[1], w[2], w[3]);
        codes[2 * static_cast<int64_t>(idx) + 1] = make_uint4(w[4], w[5], w[6], w[7]);
        const int line = idx >> log2_nblk, kb = idx & (nblk - 1);
        const int mat = line / rows_per_mat, r = line - mat * rows_per_mat;
        const int64_t tile = static_cast<int64_t>(mat) * n_tiles + (r >> 7);
        scales[tile * kAtomBytes + atom_offset(r & (kTile - 1), kb)] = static_cast<uint8_t>(X + 127);
        if (norm_mode != NORM_NONE) {
            // the nblk blocks of a row sit in nblk consecutive lanes (the
            // warp's indices are consecutive, nblk divides 32, total is a
            // multiple of nblk); the lanes of this pass are those below total
            const int left = total - (idx - static_cast<int>(threadIdx.x & 31));
            const unsigned act = left >= 32 ? 0xFFFFFFFFu : (1u << left) - 1u;
            float ss = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) ss = sumsq_e4m3x4(w[i], ss);
            const float p2 = pow2f(X);
            ss = ss * p2 * p2;
            for (int o = 1; o < nblk; o <<= 1) ss += __shfl_xor_sync(act, ss, o);
            const float bnd = norm_bound(ss);  // every lane of the row holds it
            if (norm_mode == NORM_ROW) {
                if (kb == 0) norms[line] = bnd;
            } else {
                // one atomic per KV tile and warp: the lanes of a tile take
                // their maximum first (non-negative floats order like their
                // bit patterns)
                const unsigned grp = __match_any_sync(act, tile);
                const unsigned m = __reduce_max_sync(grp, __float_as_uint(bnd));
                if ((threadIdx.x & 31) == __ffs(grp) - 1)
                    atomicMax(reinterpret_cast<unsigned int*>(norms + tile), m);
            }
        }
    }
}

// V of the fused attention (blocks of 32 keys along the keys, output
// transposed: codes [batch][cols][pitch] with the keys contiguous), one
// 128-key tile of one head per CTA and a thread per column pair and 32-key
// block: the tile's codes are assembled in shared memory ([column][key], rows
// padded to 144 bytes against bank conflicts) and written out as whole
// 128-byte lines, one per column, rather than as 32-byte pieces of 32
// different lines per store.  A warp's loads read 128 contiguous bytes of a
// key row each.  Keys in [rows, pitch) get zero codes (loaded as zeros).
template <int kElem>
__global__ void __launch_bounds__(256) quant_cols_attn_kernel(
    const uint32_t* __restrict__ x, int rows, int log2_cpairs, uint8_t* __restrict__ codes,
    int pitch, uint8_t* __restrict__ scales) {
    __shared__ __align__(16) uint8_t tile[128][144];
    const int cpairs = 1 << log2_cpairs;  // D / 2 = 32 or 64
    const int cols = 2 * cpairs;
    const int n_tiles = gridDim.x;
    const int rt = blockIdx.x;            // key tile
    const int64_t b = blockIdx.y;         // head
    const int cp = threadIdx.x & (cpairs - 1);
    const int kb = threadIdx.x >> log2_cpairs;  // 32-key block of the tile (blockDim = 4 cpairs)
    const int r0 = rt * kTile + 32 * kb;
    if (r0 < rows) {
        const uint32_t* src = x + (b * rows + r0) * cpairs + cp;
        uint32_t w[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) w[j] = r0 + j < rows ? __ldg(src + static_cast<int64_t>(j) * cpairs) : 0u;
        uint32_t u0[16], u1[16];  // columns 2 cp and 2 cp + 1 as pairs of keys (2j, 2j + 1)
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            u0[j] = __byte_perm(w[2 * j], w[2 * j + 1], 0x5410);
            u1[j] = __byte_perm(w[2 * j], w[2 * j + 1], 0x7632);
        }
        const int64_t atom = (b * n_tiles + rt) * kAtomBytes;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t q[8];
            const int X = quantize_block_attn<kElem>(h ? u1 : u0, q);
            const int c = 2 * cp + h;
            uint4* d4 = reinterpret_cast<uint4*>(&tile[c][32 * kb]);
            d4[0] = make_uint4(q[0], q[1], q[2], q[3]);
            d4[1] = make_uint4(q[4], q[5], q[6], q[7]);
            scales[atom + atom_offset(c, kb)] = static_cast<uint8_t>(X + 127);
        }
    }
    __syncthreads();
    // the tile's part of each line: up to 128 bytes, a multiple of 16 (pitch
    // and the tile start are), 8 threads per line
    const int valid = min(kTile, pitch - rt * kTile) >> 4;
    for (int i = threadIdx.x; i < cols * 8; i += blockDim.x) {
        const int c = i >> 3, k = i & 7;
        if (k < valid)
            *reinterpret_cast<uint4*>(codes + (b * cols + c) * static_cast<int64_t>(pitch) + rt * kTile + 16 * k) =
                *reinterpret_cast<const uint4*>(&tile[c][16 * k]);
    }
}

}  // namespace

cudaError_t launch_quant_rows(const uint16_t* x, int64_t lines, int64_t cols, int elem, int layout,
                              uint8_t* codes, uint8_t* scales, int64_t rows_per_mat,
                              cudaStream_t st, float* norms, int norm_mode) {
    const int64_t total = lines * ((cols + 31) / 32);
    if (total == 0) return cudaSuccess;
    // row norms need the ATTN layout and whole rows of 2 or 4 blocks in a warp
    if (norm_mode != NORM_NONE && (layout != QL_ATTN || !norms || (cols != 64 && cols != 128)))
        return cudaErrorInvalidValue;
    const int vec = (cols % 8 == 0) && ((reinterpret_cast<uintptr_t>(x) & 15) == 0) &&
                    ((reinterpret_cast<uintptr_t>(codes) & 15) == 0);
    int dev = 0, nsm = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    const int threads = 256;
    const int64_t rpm = rows_per_mat > 0 ? rows_per_mat : lines;
    if (layout == QL_ATTN && vec && (cols == 64 || cols == 128) && total < (int64_t{1} << 31) &&
        rpm < (int64_t{1} << 31)) {
        // the fused attention's operands: specialised kernel, 32-bit indexing
        int64_t blocks = (total + threads - 1) / threads;
        blocks = blocks < static_cast<int64_t>(nsm) * 8 ? blocks : static_cast<int64_t>(nsm) * 8;
        const int l2 = cols == 128 ? 2 : 1;
        const uint4* x4 = reinterpret_cast<const uint4*>(x);
        uint4* c4 = reinterpret_cast<uint4*>(codes);
        const int ln = static_cast<int>(lines), rp = static_cast<int>(rpm);
        if (elem == ELEM_E4M3)
            quant_rows_attn_kernel<ELEM_E4M3><<<static_cast<unsigned>(blocks), threads, 0, st>>>(
                x4, ln, l2, rp, c4, scales, norms, norm_mode);
        else if (elem == ELEM_E2M3)
            quant_rows_attn_kernel<ELEM_E2M3><<<static_cast<unsigned>(blocks), threads, 0, st>>>(
                x4, ln, l2, rp, c4, scales, norms, norm_mode);
        else
            quant_rows_attn_kernel<ELEM_E2M1><<<static_cast<unsigned>(blocks), threads, 0, st>>>(
                x4, ln, l2, rp, c4, scales, norms, norm_mode);
        return cudaGetLastError();
    }
    int64_t blocks = (total + threads - 1) / threads;
    blocks = blocks < static_cast<int64_t>(nsm) * 16 ? blocks : static_cast<int64_t>(nsm) * 16;
    quant_rows_kernel<<<static_cast<unsigned>(blocks), threads, 0, st>>>(
        x, lines, cols, elem, layout, codes, scales, rows_per_mat > 0 ? rows_per_mat : lines, vec,
        norms, norm_mode);
    return cudaGetLastError();
}

cudaError_t launch_quant_cols(const uint16_t* x, int64_t batch, int64_t rows, int64_t cols,
                              int elem, int layout, uint8_t* codes, int64_t code_pitch,
                              uint8_t* scales, cudaStream_t st) {
    if (batch == 0 || rows == 0 || cols == 0) return cudaSuccess;
    if (layout == QL_ATTN && (cols == 64 || cols == 128) && (reinterpret_cast<uintptr_t>(x) & 15) == 0 &&
        (reinterpret_cast<uintptr_t>(codes) & 15) == 0 && code_pitch % 16 == 0 &&
        code_pitch < (int64_t{1} << 31) && batch <= 65535 && rows < (int64_t{1} << 31) - kTile) {
        // the fused attention's V operand: a CTA per 128-key tile and head, a
        // thread per column pair and 32-key block
        const uint32_t* x2 = reinterpret_cast<const uint32_t*>(x);
        const int r = static_cast<int>(rows), pt = static_cast<int>(code_pitch);
        const int l2 = cols == 128 ? 6 : 5;
        const dim3 grid(static_cast<unsigned>((rows + kTile - 1) / kTile), static_cast<unsigned>(batch));
        const unsigned threads = 4u << l2;  // 4 blocks of 32 keys x column pairs
        if (elem == ELEM_E4M3)
            quant_cols_attn_kernel<ELEM_E4M3><<<grid, threads, 0, st>>>(x2, r, l2, codes, pt, scales);
        else if (elem == ELEM_E2M3)
            quant_cols_attn_kernel<ELEM_E2M3><<<grid, threads, 0, st>>>(x2, r, l2, codes, pt, scales);
        else
            quant_cols_attn_kernel<ELEM_E2M1><<<grid, threads, 0, st>>>(x2, r, l2, codes, pt, scales);
        return cudaGetLastError();
    }
    dim3 grid(static_cast<unsigned>((rows + 31) / 32),
              static_cast<unsigned>((cols + kColTileC - 1) / kColTileC),
              static_cast<unsigned>(batch));
    quant_cols_kernel<<<grid, 256, 0, st>>>(x, rows, cols, elem, layout, codes, code_pitch, scales);
    return cudaGetLastError();
}

}  // namespace fsa
