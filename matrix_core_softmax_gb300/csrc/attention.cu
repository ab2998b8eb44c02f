// attention.cu -- Fused-Softmax MX attention forward for sm_103a.
//
// Method ("Fused-Softmax shifts an AI attention bottleneck onto faster GPU
// hardware", paragraphs 5-8; "Fused softmax makes quantized attention faster
// on AMD GPUs", "What the evidence shows", bullet "Move work, keep
// correction"):
//   * S = Q^ K^T on block-scaled tensor cores (tcgen05 kind::mxf8f6f4, E8M0
//     scales in TMEM, FP32 accumulator in TMEM);
//   * the reference maximum of each row is frozen at KV tile 0 and the
//     Schraudolph affine map y = alpha * S + beta (alpha = 128 log2(e) sm,
//     beta = 128*127 - 7 - alpha * m) is applied to the accumulator with one
//     FMA per score;
//   * the rounded y, clamped to [0, 0x7F7F], IS a bf16 bit pattern (integer
//     reinterpretation); each 32-key block of those bf16 weights gets its
//     E8M0 scale and is converted to the P element type (two-stage
//     conversion);
//   * O += P^ V^ and l += P^ 1 come from one more block-scaled MMA on the
//     same P^, read from tensor memory: the V^T operand carries 16 extra
//     all-ones rows, so column D of the accumulator is the row sum;
//   * a row whose tile maximum passes its reference by more than theta
//     rolls back: O and l are rescaled by exp(m_old - m_new) in TMEM and the
//     reference moves to the tile maximum ("recovery procedure", paragraph 5).
//
// Work decomposition: one CTA per (128-row query tile, head); 12 warps:
//   warps 0-3  softmax warpgroup 0: KV tiles 0, 2, 4, ... (S buffer 0, P buffer 0)
//   warps 4-7  softmax warpgroup 1: KV tiles 1, 3, 5, ... (S buffer 1, P buffer 1)
//              thread r of a warpgroup owns query row r = TMEM lane r; the
//              tile maxima are handed from one warpgroup to the other
//              (shared memory + mbarrier) and each replays the gate;
//   warp 8     TMA producer of Q and the K ring; warp 10 of the V^T ring;
//   warp 9     TMEM allocator and issuer of the score products;
//   warp 11    issuer of the PV products.
// The score product of tile t+1 runs while tile t is converted, and each
// scheduler holds two softmax warps.  Each tile's scores are read from TMEM
// once; P and its scale bytes go back to TMEM with tcgen05.st.
//
// MMA operands are E4M3 bit patterns for all three formats: every E2M3 and
// E2M1 value is exactly an E4M3 value, kind::mxf8f6f4 runs at one rate for
// all of these types, and a six-bit P block with scale 2^X is stored as the
// E4M3 pattern of p / 2^(X+6) with scale byte X + 6 + 127 (E2M3's grid is
// E4M3's grid shifted by 2^6 from its subnormal step up to its maximum).
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>

#include "fsa_internal.h"
#include "sm100_ptx.cuh"

namespace fsa {
namespace {

constexpr int kStages = 3;
constexpr int kPBuf = 2;  // P buffers in TMEM: the CTA's tile g uses g % 2 (one per warpgroup)
constexpr int kThreads = 384;  // 2 softmax warpgroups + (K loader, MMA, V loader, spare)
constexpr int kWarpLoad = 8, kWarpMma = 9, kWarpLoadV = 10, kWarpPv = 11;
// Register split: launched at 168 per thread (384 x 168 = 64512), the helper
// warpgroup gives back to 32 and the softmax warpgroups take 232:
// 2 * 128 * 232 + 128 * 32 = 63488 <= 64512.
constexpr int kLaunchRegs = 168, kSoftmaxRegs = 232, kHelperRegs = 32;
static_assert(2 * 128 * kSoftmaxRegs + 128 * kHelperRegs <= kThreads * kLaunchRegs,
              "register split exceeds the launch allocation");
// Work items of at most this many KV tiles go to the persistent kernel
// (measured on GB300 with 75600 query rows x 40 heads: faster up to 2048
// keys, even at 4096, slower at 8192), whatever the number of items.
constexpr int kPersistentMaxTiles = 16;
// The EFQ producer's persistent kernel also wins at 64 and 128 KV tiles per
// item (B=1 H=16 S=8192: 1248 -> 1335 TFLOP/s; H=32 S=16384: 1460 -> 1506)
// and loses at 591 (1758 -> 1687).
constexpr int kPersistentMaxTilesEfq = 128;
// The persistent kernel's helper warps keep the rings' state across work
// items and give back only to 40: 2 * 128 * 232 + 128 * 40 = 64512.
constexpr int kHelperRegsPersistent = 40;
static_assert(2 * 128 * kSoftmaxRegs + 128 * kHelperRegsPersistent <= kThreads * kLaunchRegs,
              "register split exceeds the launch allocation");
constexpr int kTileBytes = 128 * 128;  // one 128 x 128 byte operand tile
constexpr int kVBytes = kTileBytes + 16 * 128;  // V^T tile + 16 all-ones rows (row sums)
constexpr uint32_t kTmemCols = 512;
// TMEM column map: S0, S1 (128 each), O (D columns) with l in column D of
// the same accumulator (D + 16 columns written), P0, P1 (32 each: 128 E4M3
// bytes per row), and the scale-factor atoms (4 columns per atom)
constexpr uint32_t kColS0 = 0, kColO = 256;  // S1 = kColS0 + 128, l = kColO + D
constexpr uint32_t kColP = 400;              // + 32 * (g & 1)
constexpr uint32_t kColSfQ = 464, kColSfK = 468 /* +4*(g&1) */, kColSfP = 476 /* +4*(g&1) */,
                   kColSfV = 484 /* +8*(g&1): V rows 0-127, then unit scales for rows 128-255 */,
                   kColSfQ1 = 500 /* persistent kernel: scales of Q buffer 1 */;
static_assert(kColSfV + 16 <= kColSfQ1 && kColSfQ1 + 4 <= 512, "TMEM column map beyond the allocation");
constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23: x + kMagic holds rne(x) in its low bits

struct __align__(1024) Smem {
    uint8_t q[2][kTileBytes];  // Q tile (persistent kernel: of its item j in buffer j % 2)
    uint8_t k[kStages][kTileBytes];
    uint8_t v[kStages][kVBytes];  // rows [0, D): V^T tile; rows [D, D+16): all ones
    uint8_t q_sf[2][kAtomBytes];
    uint8_t k_sf[kStages][kAtomBytes];
    uint8_t v_sf[kStages][kAtomBytes];
    uint8_t ones_sf[kAtomBytes];
    float tmax_x[8][128];  // row maxima of the CTA's tile g in slot g % 8, read by the other warpgroup
    uint64_t bar_q[2];    // Q tile of buffer i landed
    uint64_t q_empty[2];  // persistent kernel: score products of the item in Q buffer i retired
    uint64_t k_full[kStages];   // K tile landed
    uint64_t k_empty[kStages];  // score product that read the K tile retired
    uint64_t v_full[kStages];
    uint64_t v_empty[kStages];  // PV product that read the V tile retired
    uint64_t s_full[2];
    uint64_t s_free[2];
    uint64_t p_full[kPBuf];
    uint64_t p_free[kPBuf];  // PV of the tile that used P buffer i (and its scales) retired
    uint64_t m_ready[8]; // slot i of tmax_x written (tiles i, i + 8, ...)
    uint64_t o_full;  // the (item's) last PV product retired
    uint64_t o_free;  // persistent kernel: the item's O and l read by the epilogue (8 softmax warps)
    uint64_t drain_qk, drain_pv;
    uint32_t tmem_base;
    int abort;
};

static_assert(sizeof(Smem) <= 232448, "shared memory beyond the 227 KB a CTA may use");

struct Params {
    const uint8_t* q_sf;
    const uint8_t* k_sf;
    const uint8_t* v_sf;
    const float* q_norm;  // six-bit P: [BH][Sq] bounds of |q^_i|
    const float* k_norm;  // six-bit P: [BH][n_t] per KV tile, bound of max_j |k^_j|
    __nv_bfloat16* o;
    uint8_t* rollback_bits;
    unsigned long long* rollback_count;
    unsigned int* err_word;
    int Sq, Sk, D, n_t;  // query rows, keys, head dim, KV tiles ceil(Sk / 128)
    int n_qt, n_items;   // query tiles ceil(Sq / 128); work items n_qt * B * H
    float sm_scale;  // s = sm_scale * accumulator
    float alpha;     // 128 * log2(e) * sm_scale
    float theta;     // gate threshold, natural-log score units
    float theta_raw; // theta / sm_scale: the same threshold on accumulator values
    int sb_theta;    // shortcut gate: the P block scale byte of theta's own weight code
    uint64_t timeout_ns;
    int debug_flags;
    // 2^8 and 2^16, held in registers: byte and half-word packing as an
    // integer multiply-add runs on the FMA pipe, while a constant multiplier
    // would become a shift on the integer ALU, the softmax warps' busiest pipe
    uint32_t mul8, mul16;
    uint32_t mul4;  // 2^4, the same for the EFQ code nibbles
    // EFQ producer: c = sm_scale * log2(e); code = clip(floor((r - tau) / h), 0, 7)
    float efq_c, efq_a8, efq_inv8h, efq_tau;  // a8 = c / (8 h), inv8h = 1 / (8 h)
};

// P producer of a kernel instance: the method's Schraudolph code and
// two-stage conversion to E4M3 (MXFP8) or six-bit E2M3 (MXFP6, MXFP4) with
// the frozen reference and rollback gate, or the EFQ-Softmax E2M1 producer
// with the running row maximum.
enum PProducer : int { kPE4M3 = 0, kPE2M3 = 1, kPEfq = 2 };

__device__ __forceinline__ void raise_abort(Smem& sm, const Params& p) {
    sm.abort = 1;
    atomicOr(p.err_word, kErrTimeout);
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
__device__ __forceinline__ float fmin3(float a, float b, float c) {
    float d;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Max and min of 32 raw scores (three-input max/min in a depth-4 tree, so the
// reductions do not serialise on instruction latency).
__device__ __forceinline__ void maxmin32(const uint32_t (&v)[32], float& mx, float& mn) {
    float a[11], b[11];
#pragma unroll
    for (int i = 0; i < 10; ++i) {
        a[i] = fmax3(__uint_as_float(v[3 * i]), __uint_as_float(v[3 * i + 1]), __uint_as_float(v[3 * i + 2]));
        b[i] = fmin3(__uint_as_float(v[3 * i]), __uint_as_float(v[3 * i + 1]), __uint_as_float(v[3 * i + 2]));
    }
    a[10] = fmaxf(__uint_as_float(v[30]), __uint_as_float(v[31]));
    b[10] = fminf(__uint_as_float(v[30]), __uint_as_float(v[31]));
    const float a0 = fmax3(a[0], a[1], a[2]), a1 = fmax3(a[3], a[4], a[5]), a2 = fmax3(a[6], a[7], a[8]);
    const float b0 = fmin3(b[0], b[1], b[2]), b1 = fmin3(b[3], b[4], b[5]), b2 = fmin3(b[6], b[7], b[8]);
    mx = fmax3(fmax3(a0, a1, a2), a[9], a[10]);
    mn = fmin3(fmin3(b0, b1, b2), b[9], b[10]);
}

// Maximum of 32 raw scores (three-input max in a depth-4 tree).
__device__ __forceinline__ float max32(const uint32_t (&v)[32]) {
    float a[11];
#pragma unroll
    for (int i = 0; i < 10; ++i)
        a[i] = fmax3(__uint_as_float(v[3 * i]), __uint_as_float(v[3 * i + 1]), __uint_as_float(v[3 * i + 2]));
    a[10] = fmaxf(__uint_as_float(v[30]), __uint_as_float(v[31]));
    return fmax3(fmax3(fmax3(a[0], a[1], a[2]), fmax3(a[3], a[4], a[5]), fmax3(a[6], a[7], a[8])), a[9],
                 a[10]);
}

// Minimum of 32 raw scores (three-input min in a depth-4 tree).
__device__ __forceinline__ float min32(const uint32_t (&v)[32]) {
    float a[11];
#pragma unroll
    for (int i = 0; i < 10; ++i)
        a[i] = fmin3(__uint_as_float(v[3 * i]), __uint_as_float(v[3 * i + 1]), __uint_as_float(v[3 * i + 2]));
    a[10] = fminf(__uint_as_float(v[30]), __uint_as_float(v[31]));
    return fmin3(fmin3(fmin3(a[0], a[1], a[2]), fmin3(a[3], a[4], a[5]), fmin3(a[6], a[7], a[8])), a[9],
                 a[10]);
}

// Keys at or beyond n_valid (relative to this 32-key chunk) become -inf.
__device__ __forceinline__ void mask32(uint32_t (&v)[32], int n_valid) {
#pragma unroll
    for (int j = 0; j < 32; ++j)
        if (j >= n_valid) v[j] = 0xFF800000u;
}

constexpr int kMagicBits = 0x4B400000;  // bit pattern of kMagic

// Two-stage conversion of 32 scores of one 32-key block: bf16 weight code
// (integer reinterpretation) -> E4M3 pattern of p * inv, inv = 2^-(X+off).
// Writes 8 words, element i in byte i % 4 of word i / 4.  The low 16 bits
// of y + kMagic are the code, so (y + kMagic) * 2^16 (mod 2^32) is the bf16
// weight as an FP32 pattern.
template <bool kClamp>
__device__ __forceinline__ void convert32(const uint32_t (&v)[32], float alpha, float beta,
                                          float inv, uint32_t mul16, uint32_t (&w)[8]) {
    const float2 a2 = make_float2(alpha, alpha), b2 = make_float2(beta, beta);
    const float2 m2 = make_float2(kMagic, kMagic), i2 = make_float2(inv, inv);
    float2 q[2];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        float2 y = __ffma2_rn(make_float2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])),
                              a2, b2);
        if (kClamp) {
            y.x = fmaxf(y.x, 0.0f);
            y.y = fmaxf(y.y, 0.0f);
        }
        y = __fadd2_rn(y, m2);
        const float2 pw = make_float2(__uint_as_float(__float_as_uint(y.x) * mul16),
                                      __uint_as_float(__float_as_uint(y.y) * mul16));
        q[i & 1] = __fmul2_rn(pw, i2);
        if (i & 1) w[i >> 1] = cvt_e4m3x4(q[0].x, q[0].y, q[1].x, q[1].y);
    }
}

// E4M3 P when every score of the 32-key block converts to an E4M3 normal
// (p / 2^X >= 2^-6): then the E4M3 pattern of bf16(code) / 2^X is linear in
// the integer code, rne((code - 128 X - 15360) / 16) -- 15360 = 120 << 7
// re-biases the exponent from bf16 (127) to E4M3 (7) and the division drops
// four of the seven mantissa bits with round-to-nearest-even.  Two FP32 adds
// perform both roundings: + 1.5 * 2^23 rounds y to the integer code, then
// + kx (= 1.5 * 2^27 - 1.5 * 2^23 - 15360 - 128 X, a multiple of 16) lands
// in [2^27, 2^28) where one unit in the last place is 16, rounding the
// quotient to nearest even; its pattern is 0x4D400000 + the E4M3 code.
// Packing four codes c0..c3 with integer multiply-adds only (FMA pipe):
// lo = pat1 * 2^8 + pat0 = 0x8D400000 + (c1 c0); element 2 is converted
// with kx - 16 * 0x8D40 (a multiple of 16 in the same binade, so the same
// rounding) and so has the pattern 0x4D400000 - 0x8D40 + c2, which makes
// hi = pat3 * 2^8 + pat2 = (c3 c2) - 0x8D40 (mod 2^16) in its low half;
// hi * 2^16 + lo = (c3 c2 c1 c0) exactly (mod 2^32).
__device__ __forceinline__ void convert32_linear(const uint32_t (&v)[32], float alpha, float beta,
                                                 float kx, float kx2, uint32_t mul8, uint32_t mul16,
                                                 uint32_t (&w)[8]) {
    const float2 a2 = make_float2(alpha, alpha), b2 = make_float2(beta, beta);
    const float2 m2 = make_float2(kMagic, kMagic);
    const float2 k01 = make_float2(kx, kx), k23 = make_float2(kx2, kx);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float2 y0 = __ffma2_rn(make_float2(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1])), a2, b2);
        float2 y1 = __ffma2_rn(make_float2(__uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3])), a2, b2);
        y0 = __fadd2_rn(__fadd2_rn(y0, m2), k01);
        y1 = __fadd2_rn(__fadd2_rn(y1, m2), k23);
        const uint32_t lo = __float_as_uint(y0.y) * mul8 + __float_as_uint(y0.x);
        const uint32_t hi = __float_as_uint(y1.y) * mul8 + __float_as_uint(y1.x);
        w[i] = hi * mul16 + lo;
    }
}

// P element type: E4M3 (MXFP8) or six-bit E2M3 (MXFP6, MXFP4) stored as the
// E4M3 pattern of p / 2^(X+6).  emax / mthr describe the largest element
// (1 + mthr/128) * 2^emax for the scale rule.
template <bool kE4M3> struct PType;
template <> struct PType<true> { static constexpr int kOff = 0, kEmax = 8; static constexpr uint32_t kMthr = 0x60; };
template <> struct PType<false> { static constexpr int kOff = 6, kEmax = 2; static constexpr uint32_t kMthr = 0x70; };

// E8M0 scale byte (X + 127, X including the E2M3 offset) of one 32-key
// block from its largest score.  With y = alpha * bmax + beta, y + kMagic
// holds the block's largest weight code c in its low bits (c <= 0 when the
// weight clamps to zero); the rule "smallest X with p_max <= max_elem * 2^X"
// on the bf16 pattern c (exponent field E, mantissa m) gives
// X + 127 = E - emax + (m > mthr) = floor((c + 127 - mthr) / 128) - emax,
// clamped at X = -127, which also covers every bf16 subnormal code.  y is
// clamped at -1 first so that c stays in range for any score.
template <bool kE4M3>
__device__ __forceinline__ int block_scale_byte(float bmax, float alpha, float beta) {
    using T = PType<kE4M3>;
    const float y = fmaxf(__fmaf_rn(bmax, alpha, beta), -1.0f);
    const int c = static_cast<int>(__float_as_uint(__fadd_rn(y, kMagic))) - kMagicBits;
    return max((c + 127 - static_cast<int>(T::kMthr) - 128 * T::kEmax) >> 7, 0) + T::kOff;
}

// The rollback gate of a tile whose row maximum is tmax (accumulator units)
// against the reference m.  The method's gate compares the FP32 scores: tmax
// - m > theta.  The shortcut ("Fused-Softmax shifts ...", paragraph 12: the
// fastest four-bit kernel gates on converted values and can miss a trigger)
// fires when the tile's largest P block scale under the current reference --
// the scale byte of the block holding tmax -- exceeds the scale byte of
// theta's own weight code, i.e. the FP32 gate at a threshold raised to the
// end of theta's scale binade.
template <bool kShortcut, bool kE4M3>
__device__ __forceinline__ bool gate_fires(float tmax, float m, float alpha, float theta_raw,
                                           int sb_theta) {
    if constexpr (kShortcut)
        return block_scale_byte<kE4M3>(tmax, alpha, 16249.0f - alpha * m) > sb_theta;
    else
        return tmax - m > theta_raw;
}

// E4M3 P: a block converts to E4M3 normals when its smallest code is a
// normal bf16 (>= 128) and at least 128 X + 15488 (p / 2^X >= 2^-6), with
// X = sb - 127.  Compared on the FP32 patterns of y + kMagic (signed, so a
// negative y fails).
__device__ __forceinline__ bool block_is_linear(float bn, int sb, float alpha, float beta) {
    const int cmin = static_cast<int>(__float_as_uint(__fadd_rn(__fmaf_rn(bn, alpha, beta), kMagic)));
    return cmin >= kMagicBits + 128 * max(sb - 6, 1);
}

// Six-bit P when no code of the tile is a bf16 subnormal (< 128) or falls
// below 128 (X + 1), X = sb - 127 (the scale with its E2M3 offset): then
// p / 2^X is a normal FP32 whose pattern is (code << 16) - (X << 23), one
// integer multiply-add, the same value the general path's multiply gives.
__device__ __forceinline__ bool block_is_scalable(float bn, int sb, float alpha, float beta) {
    const int cmin = static_cast<int>(__float_as_uint(__fadd_rn(__fmaf_rn(bn, alpha, beta), kMagic)));
    return cmin >= kMagicBits + 128 * max(sb - 126, 1);
}

// E2M3-in-E4M3 patterns of 32 scores with the scaling folded into the bf16
// reinterpretation: pattern(p / 2^X) = (y + kMagic) * 2^16 - X * 2^23 (mod 2^32).
__device__ __forceinline__ void convert32_scaled(const uint32_t (&v)[32], float alpha, float beta,
                                                 int sb, uint32_t mul16, uint32_t (&w)[8]) {
    const float2 a2 = make_float2(alpha, alpha), b2 = make_float2(beta, beta);
    const float2 m2 = make_float2(kMagic, kMagic);
    const uint32_t neg_x = static_cast<uint32_t>(127 - sb) << 23;  // -X * 2^23
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float2 y0 = __ffma2_rn(make_float2(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1])), a2, b2);
        float2 y1 = __ffma2_rn(make_float2(__uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3])), a2, b2);
        y0 = __fadd2_rn(y0, m2);
        y1 = __fadd2_rn(y1, m2);
        w[i] = cvt_e4m3x4(__uint_as_float(__float_as_uint(y0.x) * mul16 + neg_x),
                          __uint_as_float(__float_as_uint(y0.y) * mul16 + neg_x),
                          __uint_as_float(__float_as_uint(y1.x) * mul16 + neg_x),
                          __uint_as_float(__float_as_uint(y1.y) * mul16 + neg_x));
    }
}

// inv = 2^-X of the general conversion, X = sb - 127
__device__ __forceinline__ float general_inv(int sb) { return __int_as_float((254 - sb) << 23); }

// kx = 188728320 - 128 X: one unit of X is 8 units in the last place of a
// float in [2^27, 2^28), and 0x4D33FC40 is 188728320.0f; with X = sb - 127
// the pattern is 0x4D340038 - 8 sb.
__device__ __forceinline__ float linear_kx(int sb) { return __int_as_float(0x4D340038 - 8 * sb); }
// kx - 16 * 0x8D40 (the packing offset of every fourth element)
__device__ __forceinline__ float linear_kx2(int sb) { return __int_as_float(0x4D3372F8 - 8 * sb); }

// One arrival per warp: the lanes' preceding shared-memory writes and TMEM
// reads are ordered before lane 0's release-arrive by the warp barrier.  The
// arrive is predicated on lane 0 inside the asm, so the warp takes no
// branch (a divergent lane-0 region would cost a convergence barrier).
__device__ __forceinline__ void warp_arrive(uint64_t* bar) {
    __syncwarp();
    asm volatile("{\n.reg .pred p;\nsetp.eq.u32 p, %0, 0;\n"
                 "@p mbarrier.arrive.release.cta.shared::cta.b64 _, [%1];\n}"
                 :: "r"(threadIdx.x & 31), "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool wait_warp(uint64_t* bar, uint32_t parity, const Params& p, Smem& sm) {
    const bool w = mbar_wait(bar, parity, p.timeout_ns, &sm.abort);
    return __all_sync(0xFFFFFFFFu, w);
}

// a * b + c saturated to [0, 1] (a NaN or -inf operand gives 0)
__device__ __forceinline__ float fma_sat(float a, float b, float c) {
    float d;
    asm("fma.rn.sat.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// EFQ-Softmax codes of one 32-key block ("EFQ-Softmax: Exp-Free Quantization
// for Softmax", sections "B. Block-Scaled E2M1 Probability Representation"
// and "C. EFQ-Softmax Probability Code Generation"): with u = (s - m) c the
// shifted score in log2 units, the exponent-only scale 2^X has X = ceil(max u
// - log2 6) (the smallest X with 2^(max u) <= 6 * 2^X, 6 the largest E2M1
// value), and each residual r = u - X gives code = clip(floor((r - tau) /
// h), 0, 7).  Done as v / 8 = s * c / (8 h) + b8 saturated to [0, 1], then
// floor(8 (1 - 2^-24) v / 8) by a round-down add of 1.5 * 2^23, so that the
// low bits of the sum are the code (7 when saturated).  Four codes form a
// byte-permute selector (three integer multiply-adds) that looks the E4M3
// patterns of the E2M1 values up in two registers.  Returns X + 127.
__device__ __forceinline__ uint32_t efq_block(const uint32_t (&v)[32], float bmax, float m_acc,
                                              const Params& p, uint32_t (&w)[8]) {
    constexpr float kLog2Six = 2.5849625007211563f;
    const float xf = fminf(fmaxf(ceilf(__fmaf_rn(bmax - m_acc, p.efq_c, -kLog2Six)), -127.0f), 127.0f);
    const float b8 = __fmaf_rn(-m_acc, p.efq_a8, -(xf + p.efq_tau) * p.efq_inv8h);
    const float2 k2 = make_float2(7.99999952316284f, 7.99999952316284f);  // 8 - 2^-21
    const float2 m2 = make_float2(kMagic, kMagic);
    constexpr uint32_t kTabLo = 0x3C383000u, kTabHi = 0x4C484440u;  // E4M3 of 0, .5, 1, 1.5 | 2, 3, 4, 6
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float2 x0, x1;
        x0.x = fma_sat(__uint_as_float(v[4 * i]), p.efq_a8, b8);
        x0.y = fma_sat(__uint_as_float(v[4 * i + 1]), p.efq_a8, b8);
        x1.x = fma_sat(__uint_as_float(v[4 * i + 2]), p.efq_a8, b8);
        x1.y = fma_sat(__uint_as_float(v[4 * i + 3]), p.efq_a8, b8);
        asm("fma.rm.f32x2 %0, %0, %1, %2;" : "+l"(*reinterpret_cast<unsigned long long*>(&x0))
            : "l"(*reinterpret_cast<const unsigned long long*>(&k2)),
              "l"(*reinterpret_cast<const unsigned long long*>(&m2)));
        asm("fma.rm.f32x2 %0, %0, %1, %2;" : "+l"(*reinterpret_cast<unsigned long long*>(&x1))
            : "l"(*reinterpret_cast<const unsigned long long*>(&k2)),
              "l"(*reinterpret_cast<const unsigned long long*>(&m2)));
        // low 16 bits: code0 | code1 << 4 | code2 << 8 | code3 << 12
        const uint32_t lo = __float_as_uint(x0.y) * p.mul4 + __float_as_uint(x0.x);
        const uint32_t hi = __float_as_uint(x1.y) * p.mul4 + __float_as_uint(x1.x);
        w[i] = __byte_perm(kTabLo, kTabHi, hi * p.mul8 + lo);
    }
    return static_cast<uint32_t>(static_cast<int>(xf) + 127);
}

// The two-stage conversion of a whole tile for row r (four 32-key blocks):
// block scales from the block maxima, then the E4M3 patterns of the row in
// w0..w3 (keys 32 b .. 32 b + 31 in w_b).  Returns the four E8M0 scale bytes
// packed into a word.
template <bool kE4M3, bool kSpec>
__device__ __forceinline__ uint32_t convert_tile(const uint32_t (&s0)[32], const uint32_t (&s1)[32],
                                                 const uint32_t (&s2)[32], const uint32_t (&s3)[32],
                                                 const float (&bmax)[4], const float (&bmin)[4],
                                                 float alpha, float beta, uint32_t mul8, uint32_t mul16,
                                                 bool bounded, uint32_t (&w0)[8], uint32_t (&w1)[8],
                                                 uint32_t (&w2)[8], uint32_t (&w3)[8]) {
    const int sb0 = block_scale_byte<kE4M3>(bmax[0], alpha, beta);
    const int sb1 = block_scale_byte<kE4M3>(bmax[1], alpha, beta);
    const int sb2 = block_scale_byte<kE4M3>(bmax[2], alpha, beta);
    const int sb3 = block_scale_byte<kE4M3>(bmax[3], alpha, beta);
    if constexpr (kE4M3 && kSpec) {
        // E4M3 P: the linear conversion first (the common case), the test
        // that every element of the warp's rows is an E4M3 normal after it,
        // so the minimum tree overlaps the conversion; redone by the general
        // conversion when the test fails (rare).  (The persistent kernel
        // takes the test first: this order costs it registers.)
        convert32_linear(s0, alpha, beta, linear_kx(sb0), linear_kx2(sb0), mul8, mul16, w0);
        convert32_linear(s1, alpha, beta, linear_kx(sb1), linear_kx2(sb1), mul8, mul16, w1);
        convert32_linear(s2, alpha, beta, linear_kx(sb2), linear_kx2(sb2), mul8, mul16, w2);
        convert32_linear(s3, alpha, beta, linear_kx(sb3), linear_kx2(sb3), mul8, mul16, w3);
        if (!__all_sync(0xFFFFFFFFu, block_is_linear(fminf(fminf(bmin[0], bmin[1]), fminf(bmin[2], bmin[3])),
                                                     max(max(sb0, sb1), max(sb2, sb3)), alpha, beta))) {
            convert32<true>(s0, alpha, beta, general_inv(sb0), mul16, w0);
            convert32<true>(s1, alpha, beta, general_inv(sb1), mul16, w1);
            convert32<true>(s2, alpha, beta, general_inv(sb2), mul16, w2);
            convert32<true>(s3, alpha, beta, general_inv(sb3), mul16, w3);
        }
        return (static_cast<uint32_t>(sb0) + static_cast<uint32_t>(sb1) * mul8) +
               (static_cast<uint32_t>(sb2) + static_cast<uint32_t>(sb3) * mul8) * mul16;
    }
    // one decision for the whole tile: every row of the warp converts
    // linearly (the common case for MXFP8), else block by block.  Checked
    // once per row against the largest block threshold (sb grows with the
    // block maximum), which implies every block's own condition.
    if (kE4M3 && __all_sync(0xFFFFFFFFu, block_is_linear(fminf(fminf(bmin[0], bmin[1]), fminf(bmin[2], bmin[3])),
                                                         max(max(sb0, sb1), max(sb2, sb3)), alpha, beta))) {
        convert32_linear(s0, alpha, beta, linear_kx(sb0), linear_kx2(sb0), mul8, mul16, w0);
        convert32_linear(s1, alpha, beta, linear_kx(sb1), linear_kx2(sb1), mul8, mul16, w1);
        convert32_linear(s2, alpha, beta, linear_kx(sb2), linear_kx2(sb2), mul8, mul16, w2);
        convert32_linear(s3, alpha, beta, linear_kx(sb3), linear_kx2(sb3), mul8, mul16, w3);
    } else if (!kE4M3 && (bounded || __all_sync(0xFFFFFFFFu,
                                                block_is_scalable(fminf(fminf(bmin[0], bmin[1]), fminf(bmin[2], bmin[3])),
                                                                  max(max(sb0, sb1), max(sb2, sb3)), alpha, beta)))) {
        // six-bit P, the common case: scaling folded into the reinterpretation
        // (bounded: the warp's norm bound already proves the condition)
        convert32_scaled(s0, alpha, beta, sb0, mul16, w0);
        convert32_scaled(s1, alpha, beta, sb1, mul16, w1);
        convert32_scaled(s2, alpha, beta, sb2, mul16, w2);
        convert32_scaled(s3, alpha, beta, sb3, mul16, w3);
    } else if (kE4M3 || __any_sync(0xFFFFFFFFu,
                                   __fmaf_rn(fminf(fminf(bmin[0], bmin[1]), fminf(bmin[2], bmin[3])),
                                             alpha, beta) < 0.0f)) {
        // some weight of the warp's rows clamps to zero
        convert32<true>(s0, alpha, beta, general_inv(sb0), mul16, w0);
        convert32<true>(s1, alpha, beta, general_inv(sb1), mul16, w1);
        convert32<true>(s2, alpha, beta, general_inv(sb2), mul16, w2);
        convert32<true>(s3, alpha, beta, general_inv(sb3), mul16, w3);
    } else {
        convert32<false>(s0, alpha, beta, general_inv(sb0), mul16, w0);
        convert32<false>(s1, alpha, beta, general_inv(sb1), mul16, w1);
        convert32<false>(s2, alpha, beta, general_inv(sb2), mul16, w2);
        convert32<false>(s3, alpha, beta, general_inv(sb3), mul16, w3);
    }
    // four bytes < 256 into one word
    return (static_cast<uint32_t>(sb0) + static_cast<uint32_t>(sb1) * mul8) +
           (static_cast<uint32_t>(sb2) + static_cast<uint32_t>(sb3) * mul8) * mul16;
}

// Six-bit P without block minima.  The scaled conversion (convert32_scaled)
// is exact when every code c of the row's tile satisfies c >= 128 and
// c >= 128 (X_max + 1), X_max the largest block exponent with its E2M3 offset
// (block_is_scalable).  From the scale rule, X_max + 1 = max(floor((C - 241)
// / 128), 0) - 120 for the row's largest code C, so both hold when
// C - c_min <= 15601 and c_min >= 128.  Every code lies within 0.51 of
// alpha (acc - m) + 16249 (FP32 rounding of beta and of the FMA, then the
// rounding to an integer), and by Cauchy-Schwarz every accumulator of row i,
// the reference m among them (it is one), lies in [-A, A] with
// A = |q^_i| max_j |k^_j|.  Hence 2 |alpha| A <= 15000 gives C - c_min <=
// 15001.1 and c_min >= 16249 - 15000.6: the minima need not be taken.  The
// norm bounds come from the quantizer with a relative slack of 2^-10, and the
// 4 % margin to 15601 covers the MMA's accumulation error.  A warp takes the
// shortcut when all 32 of its rows pass (a NaN or infinite bound fails).
constexpr float kBoundLimit = 15000.0f;

__device__ __forceinline__ bool warp_bounded(const Params& p, int bh, bool row_valid, int64_t grow) {
    // the head's largest key-row bound: lane l scans tiles l, l + 32, ...;
    // non-negative floats (and +inf, NaN) compare like their bit patterns
    const float* kn = p.k_norm + static_cast<int64_t>(bh) * p.n_t;
    unsigned km = 0;
    for (int i = threadIdx.x & 31; i < p.n_t; i += 32) km = max(km, __float_as_uint(kn[i]));
    km = __reduce_max_sync(0xFFFFFFFFu, km);
    const float qn = row_valid ? p.q_norm[grow] : 0.0f;  // rows past Sq hold zeros
    const float a = 2.0f * fabsf(p.alpha) * qn * __uint_as_float(km);
    return __all_sync(0xFFFFFFFFu, a <= kBoundLimit);
}

// Per-row state of a softmax thread.
struct RowState {
    float m_acc;          // frozen reference, accumulator units
    unsigned fired;       // gate firings of this row
};

// O and l of this thread's row scaled by `rescale` in TMEM (the previous
// tile's PV product has retired).
__device__ __forceinline__ void rescale_o(uint32_t lane_addr, int D, float rescale) {
    tc_fence_after();
    uint32_t rr[32];
    for (int c = 0; c < D / 32; ++c) {
        tmem_ld32(lane_addr + kColO + 32 * c, rr);
        tmem_ld_wait();
        tmem_reg_dep(rr);
#pragma unroll
        for (int j = 0; j < 32; ++j) rr[j] = __float_as_uint(__uint_as_float(rr[j]) * rescale);
        tmem_st32(lane_addr + kColO + 32 * c, rr);
    }
    uint32_t lv;
    tmem_ld1(lane_addr + kColO + D, lv);
    tmem_ld_wait();
    tmem_st1(lane_addr + kColO + D, __float_as_uint(__uint_as_float(lv) * rescale));
    tmem_st_wait();
}

// As rescale_o, with every chunk of O and l loaded before one wait (the
// score registers are free by then).
__device__ __forceinline__ void rescale_o_all(uint32_t lane_addr, int D, float rescale) {
    tc_fence_after();
    uint32_t r0[32], r1[32], r2[32], r3[32];
    uint32_t lv;
    tmem_ld32(lane_addr + kColO, r0);
    tmem_ld32(lane_addr + kColO + 32, r1);
    if (D == 128) {
        tmem_ld32(lane_addr + kColO + 64, r2);
        tmem_ld32(lane_addr + kColO + 96, r3);
    }
    tmem_ld1(lane_addr + kColO + D, lv);
    tmem_ld_wait();
    tmem_reg_dep(r0);
    tmem_reg_dep(r1);
    if (D == 128) {
        tmem_reg_dep(r2);
        tmem_reg_dep(r3);
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        r0[j] = __float_as_uint(__uint_as_float(r0[j]) * rescale);
        r1[j] = __float_as_uint(__uint_as_float(r1[j]) * rescale);
    }
    tmem_st32(lane_addr + kColO, r0);
    tmem_st32(lane_addr + kColO + 32, r1);
    if (D == 128) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            r2[j] = __float_as_uint(__uint_as_float(r2[j]) * rescale);
            r3[j] = __float_as_uint(__uint_as_float(r3[j]) * rescale);
        }
        tmem_st32(lane_addr + kColO + 64, r2);
        tmem_st32(lane_addr + kColO + 96, r3);
    }
    tmem_st1(lane_addr + kColO + D, __float_as_uint(__uint_as_float(lv) * rescale));
    tmem_st_wait();
}

// Epilogue of one row of the persistent kernel: warpgroup wg writes columns
// [wg * D/2, (wg+1) * D/2) of o = O / l as bf16, one 32-column chunk of O at
// a time.  `o_free`, when given, is released as soon as the last chunk and l
// are read from TMEM (the next work item's first PV product may then
// overwrite O while the last division and stores run).  The division is a
// multiplication by the IEEE reciprocal of l (within 1.5 units in the last
// FP32 place of O / l, before the bf16 rounding): on items of a few KV tiles
// an IEEE division per element cost a third of the item's instructions
// (measured 785 -> 1086 TFLOP/s with four tiles per item).  The one-CTA
// kernel of E4M3 P ends the same way (its epilogue took 2.8 us of a CTA's
// 42 us with 64 KV tiles when it divided: +4 % there, +1.5 % with 128
// tiles); the six-bit and EFQ one-CTA kernels divide, their main loops
// measured faster so compiled.  Which kernel a call takes depends only on
// the key length and format, so calls with the same keys compute the same
// bytes.
__device__ __forceinline__ void epilogue_chunk(const uint32_t (&rr)[32], float l, uint4* dst) {
    const float inv = __frcp_rn(l);
    uint32_t packed[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(rr[2 * j]) * inv,
                                                  __uint_as_float(rr[2 * j + 1]) * inv);
        packed[j] = *reinterpret_cast<uint32_t*>(&h2);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
        dst[j] = make_uint4(packed[4 * j], packed[4 * j + 1], packed[4 * j + 2], packed[4 * j + 3]);
}

__device__ __forceinline__ void epilogue_row(uint32_t lane_addr, int D, int wg, bool row_valid,
                                             __nv_bfloat16* o_row, uint64_t* o_free) {
    tc_fence_after();
    const int c0 = wg * (D / 64), c1 = (wg + 1) * (D / 64);  // this warpgroup's 32-column chunks
    uint32_t rr[32], lv;
    tmem_ld1(lane_addr + kColO + D, lv);
    for (int c = c0; c < c1; ++c) {
        tmem_ld32(lane_addr + kColO + 32 * c, rr);
        tmem_ld_wait();
        tmem_reg_dep(rr);
        if (c + 1 == c1 && o_free) {
            tc_fence_before();
            warp_arrive(o_free);
        }
        if (row_valid)
            epilogue_chunk(rr, __uint_as_float(lv), reinterpret_cast<uint4*>(o_row + 32 * c));
    }
}

// One KV tile t (the it-th of warpgroup wg) for query row r: read the 128
// scores once (one TMEM wait), release the S buffer, block max/min, the
// reference hand-off and the gate (with the O / l rescale on a rollback),
// then the two-stage conversion into TMEM P buffer g % 2.  A wait that gives up
// lets the tile run to its end on whatever the buffers hold (nothing is
// read or written out of bounds); the warp-wide result, false = aborted,
// ends the loop.
// Work that must come before a rescale's wait for the previous PV product
// (none in the one-CTA kernel; see the persistent kernel).
struct NoHook {
    __device__ __forceinline__ bool operator()() const { return true; }
};

template <int kP, bool kShortcut = false, bool kSpec = false, typename Hook = NoHook>
__device__ __forceinline__ bool softmax_tile(Smem& sm, const Params& p, int t, int g, int it, int wg,
                                             int r, uint32_t lane_addr, uint32_t s_col,
                                             bool row_valid, int64_t grow, bool tail, bool bounded,
                                             RowState& rs, const Hook& before_rescale = Hook()) {
    const int D = p.D;
    const int pb = g & (kPBuf - 1);
    bool ok = mbar_wait(&sm.s_full[wg], it & 1, p.timeout_ns, &sm.abort);
    tc_fence_after();
    uint32_t s0[32], s1[32], s2[32], s3[32];
    // Buffers, slots and barrier phases follow the CTA's running tile count
    // g (g = t when a CTA processes one work item); the method's tile logic
    // follows t, the tile's index within its work item.
    const int ms = (g - 1) & 7;
    const uint32_t m_par = ((g - 1) >> 3) & 1;
    const uint32_t pf_par = ((g >> 1) - 1) & 1;
    bool have_prev, have_p;
    float prev;
    // The block maxima (and minima where the conversion needs them) of the
    // row's four 32-key blocks.  The EFQ producer needs no minima; six-bit P
    // takes them only where its norm bound does not hold (and on the tail).
    float bmax[4], bmin[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    const bool need_min = kP == kPE4M3 || (kP == kPE2M3 && (!bounded || tail));
    bool extrema_done = false;
#if defined(FSA_HAVE_TMEM_REDUCE) && !defined(FSA_NO_TMEM_REDUCE)
    if (!tail) {
        // sm_103a: the reducing TMEM load returns each block's maximum with
        // its scores, so the maxima take no instruction on the CUDA cores.
        // (A second reducing load per block for the minima was measured
        // slower than the three-input minimum tree below.)
        tmem_ld32_red<true>(s_col, s0, bmax[0]);
        tmem_ld32_red<true>(s_col + 32, s1, bmax[1]);
        tmem_ld32_red<true>(s_col + 64, s2, bmax[2]);
        tmem_ld32_red<true>(s_col + 96, s3, bmax[3]);
        // while the scores travel: non-blocking looks at the other
        // warpgroup's maximum of tile t - 1 and at this tile's P buffer (PV
        // of the CTA's tile g - 2 retired); both are normally complete by now
        have_prev = t == 0 || mbar_test(&sm.m_ready[ms], m_par);
        prev = (t > 0 && have_prev) ? sm.tmax_x[ms][r] : 0.0f;
        have_p = g < kPBuf || mbar_test(&sm.p_free[pb], pf_par);
        tmem_ld_wait();
        tmem_reg_dep(s0);
        tmem_reg_dep(s1);
        tmem_reg_dep(s2);
        tmem_reg_dep(s3);
#pragma unroll
        for (int b = 0; b < 4; ++b) tmem_reg_dep1(bmax[b]);
        if (need_min) {
            bmin[0] = min32(s0);
            bmin[1] = min32(s1);
            bmin[2] = min32(s2);
            bmin[3] = min32(s3);
        }
        extrema_done = true;
    } else
#endif
    {
        tmem_ld32(s_col, s0);
        tmem_ld32(s_col + 32, s1);
        // while the scores travel: the looks at the other warpgroup's
        // maximum and at this tile's P buffer, as above
        have_prev = t == 0 || mbar_test(&sm.m_ready[ms], m_par);
        prev = (t > 0 && have_prev) ? sm.tmax_x[ms][r] : 0.0f;
        have_p = g < kPBuf || mbar_test(&sm.p_free[pb], pf_par);
        tmem_ld_wait();
        tmem_reg_dep(s0);
        tmem_reg_dep(s1);
        // the second half travels while the first is reduced (the tail tile
        // reduces after masking, below)
        tmem_ld32(s_col + 64, s2);
        tmem_ld32(s_col + 96, s3);
        if (!tail) {
            if (need_min) {
                maxmin32(s0, bmax[0], bmin[0]);
                maxmin32(s1, bmax[1], bmin[1]);
            } else {
                bmax[0] = max32(s0);
                bmax[1] = max32(s1);
            }
        }
        tmem_ld_wait();
        tmem_reg_dep(s2);
        tmem_reg_dep(s3);
    }
    // the whole tile is in registers: the next score product may reuse S
    tc_fence_before();
    warp_arrive(&sm.s_free[wg]);
    if (!extrema_done) {
        if (tail) {
            // keys >= S of a partial last tile are masked before the gate and the conversion
            const int n_valid = p.Sk - t * kTile;
            mask32(s0, n_valid);
            mask32(s1, n_valid - 32);
            mask32(s2, n_valid - 64);
            mask32(s3, n_valid - 96);
            if (need_min) {
                maxmin32(s0, bmax[0], bmin[0]);
                maxmin32(s1, bmax[1], bmin[1]);
            } else {
                bmax[0] = max32(s0);
                bmax[1] = max32(s1);
            }
        }
        if (need_min) {
            maxmin32(s2, bmax[2], bmin[2]);
            maxmin32(s3, bmax[3], bmin[3]);
        } else {
            bmax[2] = max32(s2);
            bmax[3] = max32(s3);
        }
    }
    uint32_t w0[8], w1[8], w2[8], w3[8];
    uint32_t sfw;
    if constexpr (kP == kPEfq) {
        // online attention ("EFQ-Softmax ...", section "A. Integration with
        // Online Attention"): the running row maximum, replayed over the
        // other warpgroup's maximum of tile t - 1, and O, l rescaled exactly
        // when it grows
        const float bm0 = bmax[0], bm1 = bmax[1], bm2 = bmax[2], bm3 = bmax[3];
        const float tmax = fmaxf(fmaxf(bm0, bm1), fmaxf(bm2, bm3));
        sm.tmax_x[g & 7][r] = tmax;
        warp_arrive(&sm.m_ready[g & 7]);
        if (t > 0) {
            if (!have_prev) {
                ok &= mbar_wait(&sm.m_ready[ms], m_par, p.timeout_ns, &sm.abort);
                prev = sm.tmax_x[ms][r];
            }
            rs.m_acc = (t == 1) ? prev : fmaxf(rs.m_acc, prev);
        }
        const bool grew = t > 0 && tmax > rs.m_acc;
        const float rescale = grew ? expf((rs.m_acc - tmax) * p.sm_scale) : 1.0f;
        rs.m_acc = (t == 0) ? tmax : fmaxf(rs.m_acc, tmax);
        const bool any_grew = __any_sync(0xFFFFFFFFu, grew);
        const uint32_t sb0 = efq_block(s0, bm0, rs.m_acc, p, w0);
        const uint32_t sb1 = efq_block(s1, bm1, rs.m_acc, p, w1);
        const uint32_t sb2 = efq_block(s2, bm2, rs.m_acc, p, w2);
        const uint32_t sb3 = efq_block(s3, bm3, rs.m_acc, p, w3);
        sfw = (sb0 + sb1 * p.mul8) + (sb2 + sb3 * p.mul8) * p.mul16;
        // the running maximum grows on a large share of tiles: O and l are
        // rescaled after the conversion, so that the wait for the previous
        // PV product overlaps it (P buffer first, as below)
        if (!have_p) ok &= mbar_wait(&sm.p_free[pb], pf_par, p.timeout_ns, &sm.abort);
        if (any_grew) {
            ok &= before_rescale();
            ok &= mbar_wait(&sm.p_free[(g - 1) & 1], ((g - 1) >> 1) & 1, p.timeout_ns, &sm.abort);
            rescale_o_all(lane_addr, D, rescale);
        }
    } else {
        constexpr bool kE4M3 = kP == kPE4M3;
        // a bounded six-bit warp needs only the block maxima, except on the
        // tail tile, whose masked keys take the general conversion
        const bool no_min = !kE4M3 && bounded && !tail;
        const float tmax = fmaxf(fmaxf(bmax[0], bmax[1]), fmaxf(bmax[2], bmax[3]));
        // publish this tile's row maximum for the other warpgroup in slot g % 8;
        // the reader consumes it during its tile g + 1, long before this
        // warpgroup rewrites the slot at tile g + 8: the score product of a
        // tile needs the S buffer the other warpgroup frees two tiles
        // earlier, so neither warpgroup runs more than a few tiles ahead
        sm.tmax_x[g & 7][r] = tmax;
        warp_arrive(&sm.m_ready[g & 7]);
        // frozen reference: replay the gate over the previous tile's maximum,
        // m_{t-1} = gate(m_{t-2}, tmax_{t-1}); tile 0 initialises it
        if (t > 0) {
            if (!have_prev) {
                ok &= mbar_wait(&sm.m_ready[ms], m_par, p.timeout_ns, &sm.abort);
                prev = sm.tmax_x[ms][r];
            }
            if (t == 1 || gate_fires<kShortcut, kE4M3>(prev, rs.m_acc, p.alpha, p.theta_raw, p.sb_theta))
                rs.m_acc = prev;
        }
        bool fire = false;
        float rescale = 1.0f;
        if (t == 0) {
            rs.m_acc = tmax;
        } else if (gate_fires<kShortcut, kE4M3>(tmax, rs.m_acc, p.alpha, p.theta_raw, p.sb_theta)) {
            fire = true;
            rescale = expf((rs.m_acc - tmax) * p.sm_scale);
            rs.m_acc = tmax;
        }
        // P buffer pb is free once PV of tile g - 2 retired.  Waited first: PV
        // products retire in order, so afterwards the barrier of tile g - 1's
        // buffer is past PV_{g-3} and can only be in the phase of PV_{g-1}
        // itself (PV_{g+1} needs this tile's P).
        if (!have_p) ok &= mbar_wait(&sm.p_free[pb], pf_par, p.timeout_ns, &sm.abort);
        if (__any_sync(0xFFFFFFFFu, fire)) {
            // the bitmap was zeroed before the launch: only firings are written
            if (fire && row_valid) {
                if (p.rollback_bits) p.rollback_bits[grow * p.n_t + t] = 1;
                ++rs.fired;
            }
            // recovery: once PV of the previous tile retired, O and l of the
            // firing rows are scaled by exp(m_old - m_new) in TMEM
            ok &= before_rescale();
            ok &= mbar_wait(&sm.p_free[(g - 1) & 1], ((g - 1) >> 1) & 1, p.timeout_ns, &sm.abort);
            rescale_o(lane_addr, D, rescale);
        }
        sfw = convert_tile<kE4M3, kSpec>(s0, s1, s2, s3, bmax, bmin, p.alpha, 16249.0f - p.alpha * rs.m_acc,
                                  p.mul8, p.mul16, no_min, w0, w1, w2, w3);
    }
    // the P row into TMEM (the A operand of the PV product) and its four
    // scale bytes where the product reads the scales of row r: lane r,
    // column r / 32 of the P buffer's 4-column scale atom
    tmem_st32(lane_addr + kColP + 32 * pb, w0, w1, w2, w3);
    tmem_st1(lane_addr + kColSfP + 4 * pb + (r >> 5), sfw);
    tmem_st_wait();
    tc_fence_before();
    warp_arrive(&sm.p_full[pb]);
    return __all_sync(0xFFFFFFFFu, ok);
}

template <int kP, bool kShortcut = false>
__global__ void __launch_bounds__(kThreads, 1)
    fsa_attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const Params p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // the 128-byte-swizzled TMA/MMA tiles need a 1024-byte aligned base
    if (smem_u32(smem_raw) & 1023u) {
        if (threadIdx.x == 0) atomicOr(p.err_word, kErrMisaligned);
        return;
    }
    Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int qt = blockIdx.x;
    const int bh = blockIdx.y;
    const int q0 = qt * kTile;
    const int n_qt = gridDim.x;
    const int D = p.D;
    const int nkk = D / 32;  // MMA k-steps of the score product

    // ------------------------------------------------------------- setup
    if (warp == kWarpMma) {
        tmem_alloc(&sm.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        sm.abort = 0;
        mbar_init(&sm.bar_q[0], 1);
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&sm.k_full[i], 1);
            mbar_init(&sm.k_empty[i], 1);
            mbar_init(&sm.v_full[i], 1);
            mbar_init(&sm.v_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.s_full[i], 1);
            mbar_init(&sm.s_free[i], 4);  // one arrival per softmax warp
        }
        for (int i = 0; i < 8; ++i) mbar_init(&sm.m_ready[i], 4);
        for (int i = 0; i < kPBuf; ++i) {
            mbar_init(&sm.p_full[i], 4);
            mbar_init(&sm.p_free[i], 1);
        }
        mbar_init(&sm.o_full, 1);
        mbar_init(&sm.drain_qk, 1);
        mbar_init(&sm.drain_pv, 1);
        fence_mbar_init();
    }
    if (tid < 128) {
        // 16 all-ones rows (E4M3 1.0 = 0x38) after the D rows of every V^T
        // stage, so that one PV product of N = D + 16 also yields l = P 1,
        // and a unit-scale atom (2^0 = 127) for those rows
        for (int st = 0; st < kStages; ++st)
            reinterpret_cast<uint4*>(sm.v[st] + p.D * 128)[tid] =
                make_uint4(0x38383838u, 0x38383838u, 0x38383838u, 0x38383838u);
        reinterpret_cast<uint32_t*>(sm.ones_sf)[tid] = 0x7F7F7F7Fu;
        fence_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;

    if (warp == kWarpLoad || warp == kWarpLoadV) {
        warpgroup_reg_dec<kHelperRegs>();
        // ------------------------------------------------------ producers
        // warp 8 loads Q once and the K ring, warp 10 the V^T ring; separate
        // rings let K of tile t+3 load as soon as QK_t retired, long before
        // PV_t releases V.
        if (lane == 0) {
            const bool is_k = warp == kWarpLoad;
            const uint32_t tile_bytes = static_cast<uint32_t>(kTile * D);
            if (is_k) {
                tma_prefetch_desc(&tm_q);
                tma_prefetch_desc(&tm_k);
                mbar_arrive_expect_tx(&sm.bar_q[0], tile_bytes + kAtomBytes);
                tma_load_3d(sm.q[0], &tm_q, &sm.bar_q[0], 0, q0, bh);
                bulk_load(sm.q_sf[0], p.q_sf + (static_cast<int64_t>(bh) * n_qt + qt) * kAtomBytes,
                          kAtomBytes, &sm.bar_q[0]);
            } else {
                tma_prefetch_desc(&tm_v);
            }
            uint64_t* full = is_k ? sm.k_full : sm.v_full;
            uint64_t* empty = is_k ? sm.k_empty : sm.v_empty;
            int issued = 0;
            bool ok = true;
            int st = 0;            // ring stage of tile t
            uint32_t ph = 0;       // parity of the ring's current pass
            for (int t = 0; t < p.n_t; ++t) {
                if (t >= kStages && !mbar_wait(&empty[st], ph ^ 1u, p.timeout_ns, &sm.abort)) {
                    ok = false;
                    break;
                }
                // test hook: K tile 1 never arrives
                if (!(is_k && (p.debug_flags & 1) && t == 1)) {
                    mbar_arrive_expect_tx(&full[st], tile_bytes + kAtomBytes);
                    const int64_t a = (static_cast<int64_t>(bh) * p.n_t + t) * kAtomBytes;
                    if (is_k) {
                        tma_load_3d(sm.k[st], &tm_k, &full[st], 0, t * kTile, bh);
                        bulk_load(sm.k_sf[st], p.k_sf + a, kAtomBytes, &full[st]);
                    } else {
                        tma_load_3d(sm.v[st], &tm_v, &full[st], t * kTile, 0, bh);
                        bulk_load(sm.v_sf[st], p.v_sf + a, kAtomBytes, &full[st]);
                    }
                }
                issued = t + 1;
                if (++st == kStages) {
                    st = 0;
                    ph ^= 1u;
                }
            }
            if (!ok) raise_abort(sm, p);
            if (sm.abort) {
                // let the copies still in flight land before the CTA exits
                int dummy = 0;
                if (is_k) mbar_wait(&sm.bar_q[0], 0, p.timeout_ns, &dummy);
                for (int t = max(0, issued - kStages); t < issued; ++t) {
                    if (is_k && (p.debug_flags & 1) && t == 1) continue;
                    mbar_wait(&full[t % kStages], (t / kStages) & 1, p.timeout_ns, &dummy);
                }
            }
        }
    } else if (warp == kWarpMma || warp == kWarpPv) {
        warpgroup_reg_dec<kHelperRegs>();
        // ---------------------------------------------------------- MMA
        // Two issuing threads: warp 9 the score products (into the S
        // buffers), warp 11 the PV products (into O); a late P therefore never
        // holds back the next score product.  Descriptors are built once: the
        // start-address field counts 16-byte units, so + 2 advances an
        // operand by one 32-byte K step and + 1024 by one 16 KB buffer.
        if (lane == 0) {
            constexpr uint32_t kStageUnits = kTileBytes >> 4, kVUnits = kVBytes >> 4,
                               kAtomUnits = kAtomBytes >> 4;
#define FSA_SF(kk) ((static_cast<uint32_t>(kk) << 4) | (static_cast<uint32_t>(kk) << 29))
            bool ok = true;
            if (warp == kWarpMma) {
                const uint32_t qk_swz = D == 128 ? SWZ_128B : SWZ_64B;
                const uint32_t qk_sbo = D == 128 ? 1024u : 512u;
                const uint64_t dq = smem_desc(smem_u32(sm.q[0]), 16, qk_sbo, qk_swz);
                const uint64_t dk0 = smem_desc(smem_u32(sm.k[0]), 16, qk_sbo, qk_swz);
                const uint64_t sfk0 = smem_desc(smem_u32(sm.k_sf[0]), 0, 128, SWZ_NONE);
                constexpr uint32_t id_qk = idesc_mxf8f6f4(128, 128, 0, 0, 0, 0);
                ok = mbar_wait(&sm.bar_q[0], 0, p.timeout_ns, &sm.abort);
                if (ok) {
                    tc_fence_after();
                    tc_cp_32x128b_x4(tmem + kColSfQ, smem_desc(smem_u32(sm.q_sf[0]), 0, 128, SWZ_NONE));
                }
                int st = 0;  // K ring stage of tile t
                for (int t = 0; ok && t < p.n_t; ++t) {
                    const int sb = t & 1;
                    // S buffer sb is free once the softmax of tile t - 2 read it
                    if (t >= 2 && !mbar_wait(&sm.s_free[sb], ((t - 2) >> 1) & 1, p.timeout_ns, &sm.abort)) {
                        ok = false;
                        break;
                    }
                    if (!mbar_wait(&sm.k_full[st], (t / kStages) & 1, p.timeout_ns, &sm.abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sfb = tmem + kColSfK + 4 * sb;
                    tc_cp_32x128b_x4(sfb, sfk0 + kAtomUnits * st);
                    const uint64_t bk = dk0 + kStageUnits * st;
                    const uint32_t dst = tmem + kColS0 + 128 * sb;
                    mma_mxf8f6f4(dst, dq, bk, id_qk | FSA_SF(0), tmem + kColSfQ, sfb, 0u);
                    mma_mxf8f6f4(dst, dq + 2, bk + 2, id_qk | FSA_SF(1), tmem + kColSfQ, sfb, 1u);
                    if (nkk == 4) {
                        mma_mxf8f6f4(dst, dq + 4, bk + 4, id_qk | FSA_SF(2), tmem + kColSfQ, sfb, 1u);
                        mma_mxf8f6f4(dst, dq + 6, bk + 6, id_qk | FSA_SF(3), tmem + kColSfQ, sfb, 1u);
                    }
                    tc_commit(&sm.s_full[sb]);
                    tc_commit(&sm.k_empty[st]);
                    st = st + 1 == kStages ? 0 : st + 1;
                }
            } else {
                const uint64_t dv0 = smem_desc(smem_u32(sm.v[0]), 16, 1024, SWZ_128B);
                const uint64_t sfv0 = smem_desc(smem_u32(sm.v_sf[0]), 0, 128, SWZ_NONE);
                const uint32_t id_pv = idesc_mxf8f6f4(128, D + 16, 0, 0, 0, 0);
                // unit scales for PV B rows 128-255 (the all-ones rows when D = 128)
                const uint64_t sf1 = smem_desc(smem_u32(sm.ones_sf), 0, 128, SWZ_NONE);
                tc_cp_32x128b_x4(tmem + kColSfV + 4, sf1);
                tc_cp_32x128b_x4(tmem + kColSfV + 12, sf1);
                int st = 0;  // V ring stage of tile u
                for (int u = 0; ok && u < p.n_t; ++u) {
                    const int pb = u & (kPBuf - 1);
                    if (!mbar_wait(&sm.p_full[pb], (u >> 1) & 1, p.timeout_ns, &sm.abort) ||
                        !mbar_wait(&sm.v_full[st], (u / kStages) & 1, p.timeout_ns, &sm.abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sfa = tmem + kColSfP + 4 * pb, sfb = tmem + kColSfV + 8 * (u & 1);
                    tc_cp_32x128b_x4(sfb, sfv0 + kAtomUnits * st);
                    // A = P from TMEM: 8 columns per 32-key step
                    const uint32_t ap = tmem + kColP + 32 * pb;
                    const uint64_t bv = dv0 + kVUnits * st;
                    const uint32_t acc = u > 0 ? 1u : 0u;
                    mma_mxf8f6f4_tmem_a(tmem + kColO, ap, bv, id_pv | FSA_SF(0), sfa, sfb, acc);
                    mma_mxf8f6f4_tmem_a(tmem + kColO, ap + 8, bv + 2, id_pv | FSA_SF(1), sfa, sfb, 1u);
                    mma_mxf8f6f4_tmem_a(tmem + kColO, ap + 16, bv + 4, id_pv | FSA_SF(2), sfa, sfb, 1u);
                    mma_mxf8f6f4_tmem_a(tmem + kColO, ap + 24, bv + 6, id_pv | FSA_SF(3), sfa, sfb, 1u);
                    tc_commit(&sm.v_empty[st]);
                    tc_commit(&sm.p_free[pb]);
                    st = st + 1 == kStages ? 0 : st + 1;
                }
                if (ok) tc_commit(&sm.o_full);
            }
#undef FSA_SF
            if (!ok) {
                raise_abort(sm, p);
                int dummy = 0;
                uint64_t* drain = warp == kWarpMma ? &sm.drain_qk : &sm.drain_pv;
                tc_commit(drain);  // wait until every MMA/copy this thread issued retired
                mbar_wait(drain, 0, p.timeout_ns, &dummy);
            }
        }
    } else {
        warpgroup_reg_inc<kSoftmaxRegs>();
        // ------------------------------------------------------ softmax
        // Warpgroup wg processes the KV tiles t = wg, wg + 2, ... in TMEM S
        // buffer wg and shared P buffer wg; thread r owns query row r (TMEM
        // lane r).  Tile maxima travel between the warpgroups through
        // tmax_x / m_ready; each warpgroup replays the gate over them.
        const int wg = warp >> 2;
        const int r = tid & 127;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        const uint32_t s_col = lane_addr + kColS0 + 128 * wg;
        const bool row_valid = (q0 + r) < p.Sq;
        const int64_t grow = static_cast<int64_t>(bh) * p.Sq + q0 + r;
        RowState rs{0.0f, 0u};
        bool ok = true;
        const int t_tail = (p.Sk % kTile) ? p.n_t - 1 : p.n_t;  // index of a partial last tile
        // six-bit P: a warp whose rows satisfy the norm bound skips the block minima
        bool bounded = false;
        if constexpr (kP == kPE2M3) bounded = warp_bounded(p, bh, row_valid, grow);
        for (int t = wg, it = 0; ok && t < p.n_t; t += 2, ++it)
            ok = softmax_tile<kP, kShortcut, true>(sm, p, t, t, it, wg, r, lane_addr, s_col, row_valid,
                                                   grow, t == t_tail, bounded, rs);
        if (!ok) raise_abort(sm, p);
        if (ok) {
            ok = wait_warp(&sm.o_full, 0, p, sm);
            if (!ok) raise_abort(sm, p);
        }
        if (ok) {
            // epilogue: warpgroup wg writes columns [wg * D/2, (wg+1) * D/2)
            if constexpr (kP == kPE4M3) {
                epilogue_row(lane_addr, D, wg, row_valid, p.o + grow * D, nullptr);
            } else {
                tc_fence_after();
                uint32_t lv;
                tmem_ld1(lane_addr + kColO + D, lv);
                tmem_ld_wait();
                const float l = __uint_as_float(lv);
                for (int c = wg * (D / 64); c < (wg + 1) * (D / 64); ++c) {
                    uint32_t rr[32];
                    tmem_ld32(lane_addr + kColO + 32 * c, rr);
                    tmem_ld_wait();
                    tmem_reg_dep(rr);
                    if (row_valid) {
                        uint32_t packed[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            __nv_bfloat162 h2 = __floats2bfloat162_rn(__fdiv_rn(__uint_as_float(rr[2 * j]), l),
                                                                      __fdiv_rn(__uint_as_float(rr[2 * j + 1]), l));
                            packed[j] = *reinterpret_cast<uint32_t*>(&h2);
                        }
                        uint4* dst = reinterpret_cast<uint4*>(p.o + grow * D + 32 * c);
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            dst[j] = make_uint4(packed[4 * j], packed[4 * j + 1], packed[4 * j + 2], packed[4 * j + 3]);
                    }
                }
            }
            if (p.rollback_count) {
                unsigned tot = rs.fired;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xFFFFFFFFu, tot, o);
                if (lane == 0 && tot) atomicAdd(p.rollback_count, static_cast<unsigned long long>(tot));
            }
        }
    }

    // ------------------------------------------------------------ teardown
    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}


// Persistent variant for short key sequences (few KV tiles per work item):
// one CTA per SM walks the work items, so the launch, TMEM allocation and
// barrier set-up happen once per SM, the next item's Q tile loads into the
// second Q buffer during the current item, and its first score products run
// while the current item's output is written.
template <int kP>
__global__ void __launch_bounds__(kThreads, 1)
    fsa_attn_fwd_persistent_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const Params p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // the 128-byte-swizzled TMA/MMA tiles need a 1024-byte aligned base
    if (smem_u32(smem_raw) & 1023u) {
        if (threadIdx.x == 0) atomicOr(p.err_word, kErrMisaligned);
        return;
    }
    Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int D = p.D;
    const int nkk = D / 32;  // MMA k-steps of the score product
    // Persistent CTAs: CTA c takes the work items c, c + gridDim.x, ...; item
    // i is the query tile i % n_qt of head i / n_qt, so at any time the CTAs
    // work on neighbouring query tiles of the same head (its K and V stay in
    // L2).  Every role walks the same item sequence; the per-tile buffers
    // and barrier phases follow the CTA's running tile count.

    // ------------------------------------------------------------- setup
    if (warp == kWarpMma) {
        tmem_alloc(&sm.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        sm.abort = 0;
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.bar_q[i], 1);
            mbar_init(&sm.q_empty[i], 1);
        }
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&sm.k_full[i], 1);
            mbar_init(&sm.k_empty[i], 1);
            mbar_init(&sm.v_full[i], 1);
            mbar_init(&sm.v_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.s_full[i], 1);
            mbar_init(&sm.s_free[i], 4);  // one arrival per softmax warp
        }
        for (int i = 0; i < 8; ++i) mbar_init(&sm.m_ready[i], 4);
        for (int i = 0; i < kPBuf; ++i) {
            mbar_init(&sm.p_full[i], 4);
            mbar_init(&sm.p_free[i], 1);
        }
        mbar_init(&sm.o_full, 1);
        mbar_init(&sm.o_free, 8);  // one arrival per softmax warp after its epilogue read O
        mbar_init(&sm.drain_qk, 1);
        mbar_init(&sm.drain_pv, 1);
        fence_mbar_init();
    }
    if (tid < 128) {
        // 16 all-ones rows (E4M3 1.0 = 0x38) after the D rows of every V^T
        // stage, so that one PV product of N = D + 16 also yields l = P 1,
        // and a unit-scale atom (2^0 = 127) for those rows
        for (int st = 0; st < kStages; ++st)
            reinterpret_cast<uint4*>(sm.v[st] + p.D * 128)[tid] =
                make_uint4(0x38383838u, 0x38383838u, 0x38383838u, 0x38383838u);
        reinterpret_cast<uint32_t*>(sm.ones_sf)[tid] = 0x7F7F7F7Fu;
        fence_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;

    if (warp == kWarpLoad || warp == kWarpLoadV) {
        warpgroup_reg_dec<kHelperRegsPersistent>();
        // ------------------------------------------------------ producers
        // warp 8 loads each item's Q tile (two buffers) and the K ring, warp
        // 10 the V^T ring; separate rings let K of tile g+3 load as soon as
        // QK_g retired, long before PV_g releases V.
        if (lane == 0) {
            const bool is_k = warp == kWarpLoad;
            const uint32_t tile_bytes = static_cast<uint32_t>(kTile * D);
            if (is_k) {
                tma_prefetch_desc(&tm_q);
                tma_prefetch_desc(&tm_k);
            } else {
                tma_prefetch_desc(&tm_v);
            }
            uint64_t* full = is_k ? sm.k_full : sm.v_full;
            uint64_t* empty = is_k ? sm.k_empty : sm.v_empty;
            int issued = 0;    // ring tiles issued (the CTA's running tile count)
            int q_issued = 0;  // Q tiles issued
            bool ok = true;
            int st = 0;        // ring stage of tile g
            uint32_t ph = 0;   // parity of the ring's current pass
            for (int item = blockIdx.x, j = 0; ok && item < p.n_items; item += gridDim.x, ++j) {
                const int bh = item / p.n_qt, qt = item - bh * p.n_qt;
                if (is_k) {
                    // Q buffer j % 2 is free once the score products of item j - 2 retired
                    const int qb = j & 1;
                    if (j >= 2 && !mbar_wait(&sm.q_empty[qb], ((j >> 1) - 1) & 1, p.timeout_ns, &sm.abort)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&sm.bar_q[qb], tile_bytes + kAtomBytes);
                    tma_load_3d(sm.q[qb], &tm_q, &sm.bar_q[qb], 0, qt * kTile, bh);
                    bulk_load(sm.q_sf[qb], p.q_sf + (static_cast<int64_t>(bh) * p.n_qt + qt) * kAtomBytes,
                              kAtomBytes, &sm.bar_q[qb]);
                    q_issued = j + 1;
                }
                for (int t = 0; t < p.n_t; ++t) {
                    if (issued >= kStages && !mbar_wait(&empty[st], ph ^ 1u, p.timeout_ns, &sm.abort)) {
                        ok = false;
                        break;
                    }
                    // test hook: the CTA's K tile 1 never arrives
                    if (!(is_k && (p.debug_flags & 1) && issued == 1)) {
                        mbar_arrive_expect_tx(&full[st], tile_bytes + kAtomBytes);
                        const int64_t a = (static_cast<int64_t>(bh) * p.n_t + t) * kAtomBytes;
                        if (is_k) {
                            tma_load_3d(sm.k[st], &tm_k, &full[st], 0, t * kTile, bh);
                            bulk_load(sm.k_sf[st], p.k_sf + a, kAtomBytes, &full[st]);
                        } else {
                            tma_load_3d(sm.v[st], &tm_v, &full[st], t * kTile, 0, bh);
                            bulk_load(sm.v_sf[st], p.v_sf + a, kAtomBytes, &full[st]);
                        }
                    }
                    ++issued;
                    if (++st == kStages) {
                        st = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) raise_abort(sm, p);
            if (sm.abort) {
                // let the copies still in flight land before the CTA exits
                int dummy = 0;
                for (int j = max(0, q_issued - 2); j < q_issued; ++j)
                    mbar_wait(&sm.bar_q[j & 1], (j >> 1) & 1, p.timeout_ns, &dummy);
                for (int g = max(0, issued - kStages); g < issued; ++g) {
                    if (is_k && (p.debug_flags & 1) && g == 1) continue;
                    mbar_wait(&full[g % kStages], (g / kStages) & 1, p.timeout_ns, &dummy);
                }
            }
        }
    } else if (warp == kWarpMma || warp == kWarpPv) {
        warpgroup_reg_dec<kHelperRegsPersistent>();
        // ---------------------------------------------------------- MMA
        // Two issuing threads: warp 9 the score products (into the S
        // buffers), warp 11 the PV products (into O); a late P therefore never
        // holds back the next score product.  Descriptors are built once: the
        // start-address field counts 16-byte units, so + 2 advances an
        // operand by one 32-byte K step and + 1024 by one 16 KB buffer.
        if (lane == 0) {
            constexpr uint32_t kStageUnits = kTileBytes >> 4, kVUnits = kVBytes >> 4,
                               kAtomUnits = kAtomBytes >> 4;
#define FSA_SF(kk) ((static_cast<uint32_t>(kk) << 4) | (static_cast<uint32_t>(kk) << 29))
            bool ok = true;
            if (warp == kWarpMma) {
                const uint32_t qk_swz = D == 128 ? SWZ_128B : SWZ_64B;
                const uint32_t qk_sbo = D == 128 ? 1024u : 512u;
                const uint64_t dq0 = smem_desc(smem_u32(sm.q[0]), 16, qk_sbo, qk_swz);
                const uint64_t dk0 = smem_desc(smem_u32(sm.k[0]), 16, qk_sbo, qk_swz);
                const uint64_t sfq0 = smem_desc(smem_u32(sm.q_sf[0]), 0, 128, SWZ_NONE);
                const uint64_t sfk0 = smem_desc(smem_u32(sm.k_sf[0]), 0, 128, SWZ_NONE);
                constexpr uint32_t id_qk = idesc_mxf8f6f4(128, 128, 0, 0, 0, 0);
                int g = 0;   // the CTA's running tile count
                int st = 0;  // K ring stage of tile g
                for (int item = blockIdx.x, j = 0; ok && item < p.n_items; item += gridDim.x, ++j) {
                    const int qb = j & 1;
                    if (!mbar_wait(&sm.bar_q[qb], (j >> 1) & 1, p.timeout_ns, &sm.abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sfq = tmem + (qb ? kColSfQ1 : kColSfQ);
                    tc_cp_32x128b_x4(sfq, sfq0 + kAtomUnits * qb);
                    const uint64_t dq = dq0 + kStageUnits * qb;
                    for (int t = 0; t < p.n_t; ++t, ++g) {
                        const int sb = g & 1;
                        // S buffer sb is free once the softmax of tile g - 2 read it
                        if (g >= 2 && !mbar_wait(&sm.s_free[sb], ((g - 2) >> 1) & 1, p.timeout_ns, &sm.abort)) {
                            ok = false;
                            break;
                        }
                        if (!mbar_wait(&sm.k_full[st], (g / kStages) & 1, p.timeout_ns, &sm.abort)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t sfb = tmem + kColSfK + 4 * sb;
                        tc_cp_32x128b_x4(sfb, sfk0 + kAtomUnits * st);
                        const uint64_t bk = dk0 + kStageUnits * st;
                        const uint32_t dst = tmem + kColS0 + 128 * sb;
                        mma_mxf8f6f4(dst, dq, bk, id_qk | FSA_SF(0), sfq, sfb, 0u);
                        mma_mxf8f6f4(dst, dq + 2, bk + 2, id_qk | FSA_SF(1), sfq, sfb, 1u);
                        if (nkk == 4) {
                            mma_mxf8f6f4(dst, dq + 4, bk + 4, id_qk | FSA_SF(2), sfq, sfb, 1u);
                            mma_mxf8f6f4(dst, dq + 6, bk + 6, id_qk | FSA_SF(3), sfq, sfb, 1u);
                        }
                        tc_commit(&sm.s_full[sb]);
                        tc_commit(&sm.k_empty[st]);
                        st = st + 1 == kStages ? 0 : st + 1;
                    }
                    // the item's Q buffer (and its scale copy) is read by now
                    if (ok) tc_commit(&sm.q_empty[qb]);
                }
            } else {
                const uint64_t dv0 = smem_desc(smem_u32(sm.v[0]), 16, 1024, SWZ_128B);
                const uint64_t sfv0 = smem_desc(smem_u32(sm.v_sf[0]), 0, 128, SWZ_NONE);
                const uint32_t id_pv = idesc_mxf8f6f4(128, D + 16, 0, 0, 0, 0);
                // unit scales for PV B rows 128-255 (the all-ones rows when D = 128)
                const uint64_t sf1 = smem_desc(smem_u32(sm.ones_sf), 0, 128, SWZ_NONE);
                tc_cp_32x128b_x4(tmem + kColSfV + 4, sf1);
                tc_cp_32x128b_x4(tmem + kColSfV + 12, sf1);
                int g = 0;   // the CTA's running tile count
                int st = 0;  // V ring stage of tile g
                for (int item = blockIdx.x, j = 0; ok && item < p.n_items; item += gridDim.x, ++j) {
                    // O of the previous item must have been read by the epilogue
                    if (j > 0 && !mbar_wait(&sm.o_free, (j - 1) & 1, p.timeout_ns, &sm.abort)) {
                        ok = false;
                        break;
                    }
                    for (int u = 0; u < p.n_t; ++u, ++g) {
                        const int pb = g & (kPBuf - 1);
                        if (!mbar_wait(&sm.p_full[pb], (g >> 1) & 1, p.timeout_ns, &sm.abort) ||
                            !mbar_wait(&sm.v_full[st], (g / kStages) & 1, p.timeout_ns, &sm.abort)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t sfa = tmem + kColSfP + 4 * pb, sfb = tmem + kColSfV + 8 * (g & 1);
                        tc_cp_32x128b_x4(sfb, sfv0 + kAtomUnits * st);
                        // A = P from TMEM: 8 columns per 32-key step
                        const uint32_t ap = tmem + kColP + 32 * pb;
                        const uint64_t bv = dv0 + kVUnits * st;
                        const uint32_t acc = u > 0 ? 1u : 0u;
                        mma_mxf8f6f4_tmem_a(tmem + kColO, ap, bv, id_pv | FSA_SF(0), sfa, sfb, acc);
                        mma_mxf8f6f4_tmem_a(tmem + kColO, ap + 8, bv + 2, id_pv | FSA_SF(1), sfa, sfb, 1u);
                        mma_mxf8f6f4_tmem_a(tmem + kColO, ap + 16, bv + 4, id_pv | FSA_SF(2), sfa, sfb, 1u);
                        mma_mxf8f6f4_tmem_a(tmem + kColO, ap + 24, bv + 6, id_pv | FSA_SF(3), sfa, sfb, 1u);
                        tc_commit(&sm.v_empty[st]);
                        tc_commit(&sm.p_free[pb]);
                        st = st + 1 == kStages ? 0 : st + 1;
                    }
                    if (ok) tc_commit(&sm.o_full);
                }
            }
#undef FSA_SF
            if (!ok) {
                raise_abort(sm, p);
                int dummy = 0;
                uint64_t* drain = warp == kWarpMma ? &sm.drain_qk : &sm.drain_pv;
                tc_commit(drain);  // wait until every MMA/copy this thread issued retired
                mbar_wait(drain, 0, p.timeout_ns, &dummy);
            }
        }
    } else {
        warpgroup_reg_inc<kSoftmaxRegs>();
        // ------------------------------------------------------ softmax
        // Warpgroup wg processes the tiles g with g % 2 == wg (the CTA's
        // running tile count) in TMEM S buffer wg and P buffer wg; thread r
        // owns query row r (TMEM lane r).  Tile maxima travel between the
        // warpgroups through tmax_x / m_ready; each warpgroup replays the
        // gate over them.  After an item's last PV both warpgroups write
        // half of its output and release O for the next item.
        const int wg = warp >> 2;
        const int r = tid & 127;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        const uint32_t s_col = lane_addr + kColS0 + 128 * wg;
        const int t_tail = (p.Sk % kTile) ? p.n_t - 1 : p.n_t;  // index of a partial last tile
        bool ok = true;
        int it = 0;  // tiles this warpgroup processed (phase of its S buffer)
        RowState rs{0.0f, 0u};  // the firing count runs over all items
        // The epilogue of item j - 1 is owed while item j starts: the
        // warpgroup whose first tile of item j is tile 0 converts that tile
        // first (it needs no reference, gate or rescale, so it waits on
        // nothing the owed epilogue holds back), while the last PV product of
        // item j - 1 completes; the other warpgroup writes its half first,
        // since its first tile (1) may roll back and wait for PV of tile 0,
        // which waits for both halves of the epilogue (o_free).
        bool owed = false;
        bool owed_valid = false;
        int64_t owed_grow = 0;
        for (int j = 0; ok; ++j) {
            const int item = blockIdx.x + j * gridDim.x;
            const bool have = item < p.n_items;
            const int g0 = j * p.n_t;  // running count of the item's tile 0
            const int bh = have ? item / p.n_qt : 0;
            const int q0 = have ? (item - bh * p.n_qt) * kTile : 0;
            const bool row_valid = have && (q0 + r) < p.Sq;
            const int64_t grow = static_cast<int64_t>(bh) * p.Sq + q0 + r;
            // six-bit P: a warp whose rows satisfy the norm bound skips the block minima
            bool bounded = false;
            if constexpr (kP == kPE2M3) {
                if (have) bounded = warp_bounded(p, bh, row_valid, grow);
            }
            rs.m_acc = 0.0f;
            const int t0 = (wg - g0) & 1;  // this warpgroup's first tile of the item
            // O and l of item j - 1 are released to item j's first PV product
            // as soon as they are read
            auto pay = [&]() -> bool {
                if (!owed) return true;
                const bool w = wait_warp(&sm.o_full, (j - 1) & 1, p, sm);
                if (w) epilogue_row(lane_addr, D, wg, owed_valid, p.o + owed_grow * D, &sm.o_free);
                owed = false;
                return w;
            };
            // Every warpgroup writes the epilogue it owes after its first tile
            // of item j; should that tile roll back, before its rescale's wait
            // for the item's first PV product (which waits for the epilogue).
            // Six-bit P keeps the epilogue first when its first tile is tile 1
            // (measured faster so: 1168 against 1015 TFLOP/s with four KV
            // tiles per item; E4M3 P 1270 against 1090, EFQ 995 against 956).
            constexpr bool kDeferAll = kP != kPE2M3;
            const bool defer = have && (kDeferAll ? t0 < p.n_t : t0 == 0);
            if (owed && !defer) {
                if (ok) ok = pay();
                if (!ok) break;
            }
            if (!have) break;
            for (int t = t0; ok && t < p.n_t; t += 2, ++it) {
                if constexpr (kDeferAll)
                    ok = softmax_tile<kP>(sm, p, t, g0 + t, it, wg, r, lane_addr, s_col, row_valid, grow,
                                          t == t_tail, bounded, rs, pay);
                else
                    ok = softmax_tile<kP>(sm, p, t, g0 + t, it, wg, r, lane_addr, s_col, row_valid, grow,
                                          t == t_tail, bounded, rs);
                if (owed) ok = pay() && ok;  // deferred past the first tile
            }
            owed = true;
            owed_valid = row_valid;
            owed_grow = grow;
        }
        if (!ok) raise_abort(sm, p);
        if (ok && p.rollback_count) {
            unsigned tot = rs.fired;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xFFFFFFFFu, tot, o);
            if (lane == 0 && tot) atomicAdd(p.rollback_count, static_cast<unsigned long long>(tot));
        }
    }

    // ------------------------------------------------------------ teardown
    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

cudaError_t launch_fsa_attention(const AttnLaunch& a, cudaStream_t st) {
    Params p{};
    p.q_sf = a.ws.qsf;
    p.k_sf = a.ws.ksf;
    p.v_sf = a.ws.vsf;
    p.q_norm = a.ws.qnorm;
    p.k_norm = a.ws.knorm;
    p.o = reinterpret_cast<__nv_bfloat16*>(a.o);
    p.rollback_bits = a.rollback_bits;
    p.rollback_count = a.rollback_count;
    p.err_word = a.err_word;
    p.Sq = a.Sq;
    p.Sk = a.Sk;
    p.D = a.D;
    p.n_t = (a.Sk + kTile - 1) / kTile;
    p.n_qt = (a.Sq + kTile - 1) / kTile;
    const int64_t n_items = static_cast<int64_t>(p.n_qt) * a.BH;
    if (n_items > INT32_MAX) return cudaErrorInvalidValue;
    p.n_items = static_cast<int>(n_items);
    p.sm_scale = a.sm_scale;
    p.alpha = static_cast<float>(128.0 * 1.4426950408889634 * static_cast<double>(a.sm_scale));
    p.theta = a.threshold;
    p.theta_raw = a.threshold / a.sm_scale;
    {
        // theta's own weight code and its P block scale byte (as
        // block_scale_byte computes it: E4M3 P for MXFP8, six-bit P with its
        // offset of 6 otherwise)
        const double y = 128.0 * (static_cast<double>(a.threshold) * 1.4426950408889634 + 127.0) - 7.0;
        const int c = static_cast<int>(std::nearbyint(y < 0x7F7F ? y : 0x7F7F));
        p.sb_theta = a.fmt == 0 ? std::max((c + 127 - 0x60 - 128 * 8) >> 7, 0)
                                : std::max((c + 127 - 0x70 - 128 * 2) >> 7, 0) + 6;
    }
    p.timeout_ns = a.timeout_ns;
    p.debug_flags = a.debug_flags;
    p.mul8 = 1u << 8;
    p.mul16 = 1u << 16;
    p.mul4 = 1u << 4;
    {
        const double c = static_cast<double>(a.sm_scale) * 1.4426950408889634;
        p.efq_c = static_cast<float>(c);
        p.efq_a8 = static_cast<float>(c / (8.0 * a.efq_h));
        p.efq_inv8h = static_cast<float>(1.0 / (8.0 * a.efq_h));
        p.efq_tau = a.efq_tau;
    }
    const size_t smem = sizeof(Smem);
    int dev = 0, n_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    // short key sequences: the per-CTA set-up and pipeline fill would
    // dominate a CTA that runs only a few KV tiles, so persistent CTAs (one
    // per SM, at most one per work item) walk the work items instead.  The
    // choice depends on the key length and the format alone, not on the
    // number of items, so every call with the same keys -- a whole tensor or
    // the chunks of heads of the host-buffer entry points -- takes the same
    // kernel.  The shortcut gate exists as a variant of the
    // one-CTA-per-item kernel.
    const bool shortcut = a.gate_mode == 1 && a.fmt != 3;
    const bool persistent = !shortcut && p.n_t <= (a.fmt == 3 ? kPersistentMaxTilesEfq : kPersistentMaxTiles);
    // P in E4M3 for MXFP8, six-bit E2M3 for MXFP6 and MXFP4, E2M1 codes of
    // the EFQ producer for MXFP4-EFQ
    using KernelFn = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const Params);
    KernelFn kernel;
    if (persistent)
        kernel = a.fmt == 0 ? fsa_attn_fwd_persistent_kernel<kPE4M3>
                            : (a.fmt == 3 ? fsa_attn_fwd_persistent_kernel<kPEfq>
                                          : fsa_attn_fwd_persistent_kernel<kPE2M3>);
    else if (shortcut)
        kernel = a.fmt == 0 ? fsa_attn_fwd_kernel<kPE4M3, true> : fsa_attn_fwd_kernel<kPE2M3, true>;
    else
        kernel = a.fmt == 0 ? fsa_attn_fwd_kernel<kPE4M3>
                            : (a.fmt == 3 ? fsa_attn_fwd_kernel<kPEfq> : fsa_attn_fwd_kernel<kPE2M3>);
    // the in-kernel register split assumes exactly kLaunchRegs per thread at
    // launch; anything else could make the increase wait forever
    cudaFuncAttributes fa{};
    e = cudaFuncGetAttributes(&fa, kernel);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    if (persistent) {
        const int ctas = n_items < n_sm ? static_cast<int>(n_items) : n_sm;
        kernel<<<static_cast<unsigned>(ctas), kThreads, smem, st>>>(*a.tm_q, *a.tm_k, *a.tm_v, p);
    } else {
        dim3 grid(static_cast<unsigned>(p.n_qt), static_cast<unsigned>(a.BH));
        kernel<<<grid, kThreads, smem, st>>>(*a.tm_q, *a.tm_k, *a.tm_v, p);
    }
    return cudaGetLastError();
}

}  // namespace fsa
