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
//   * O += P^ V^ and l += P^ 1 are two more block-scaled MMAs on the same
//     P^ in shared memory (l uses a 16-column all-ones B operand);
//   * a row whose tile maximum passes its reference by more than theta
//     rolls back: O and l are rescaled by exp(m_old - m_new) in TMEM and the
//     reference moves to the tile maximum ("recovery procedure", paragraph 5).
//
// Work decomposition: one CTA per (128-row query tile, head); 10 warps:
//   warps 0-3  softmax warpgroup 0: KV tiles 0, 2, 4, ... (S buffer 0, P buffer 0)
//   warps 4-7  softmax warpgroup 1: KV tiles 1, 3, 5, ... (S buffer 1, P buffer 1)
//              thread r of a warpgroup owns query row r = TMEM lane r; the
//              frozen reference is handed from one warpgroup to the other
//              after every tile (shared memory + mbarrier);
//   warp 8     TMA producer (Q once; K, V^T tiles through a 3-stage ring);
//   warp 9     TMEM allocator and the single MMA-issuing thread.
// QK^T of tile t+1 runs while tile t is converted, and each scheduler holds
// two softmax warps.  Each tile is read from TMEM twice: pass 1 takes the
// 32-key block maxima/minima (gate, block scales), pass 2 converts.
//
// MMA operands are E4M3 bit patterns for all three formats: every E2M3 and
// E2M1 value is exactly an E4M3 value, kind::mxf8f6f4 runs at one rate for
// all of these types, and a six-bit P block with scale 2^X is stored as the
// E4M3 pattern of p / 2^(X+6) with scale byte X + 6 + 127 (E2M3's grid is
// E4M3's grid shifted by 2^6 from its subnormal step up to its maximum).
#include <cuda_bf16.h>

#include "fsa_internal.h"
#include "sm100_ptx.cuh"

namespace fsa {
namespace {

constexpr int kStages = 3;
constexpr int kThreads = 320;          // 2 softmax warpgroups + loader warp + MMA warp
constexpr int kWarpLoad = 8, kWarpMma = 9;
constexpr int kTileBytes = 128 * 128;  // one 128 x 128 byte operand tile
constexpr uint32_t kTmemCols = 512;
// TMEM column map
constexpr uint32_t kColS0 = 0, kColO = 256, kColL = 384;  // S1 = kColS0 + 128
constexpr uint32_t kColSfQ = 416, kColSfK = 420 /* +4*(t&1) */, kColSfP = 428 /* +4*(u&1) */,
                   kColSfV = 436 /* +4*(u&1) */, kColSfOnes = 444;
constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23: x + kMagic holds rne(x) in its low bits

struct __align__(1024) Smem {
    uint8_t q[kTileBytes];
    uint8_t k[kStages][kTileBytes];
    uint8_t v[kStages][kTileBytes];
    uint8_t p[2][kTileBytes];
    uint8_t ones[16 * 128];
    uint8_t q_sf[kAtomBytes];
    uint8_t k_sf[kStages][kAtomBytes];
    uint8_t v_sf[kStages][kAtomBytes];
    uint8_t p_sf[2][kAtomBytes];
    uint8_t ones_sf[kAtomBytes];
    float m_ref[2][128];  // reference maximum handed from one warpgroup to the other
    uint64_t bar_q;
    uint64_t kv_full[kStages];
    uint64_t kv_empty[kStages];
    uint64_t s_full[2];
    uint64_t s_free[2];
    uint64_t p_full[2];
    uint64_t p_free[2];  // PV of the tile that used P buffer i retired
    uint64_t m_ready[2]; // warpgroup i published the reference after its tile
    uint64_t o_full;
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

static_assert(sizeof(Smem) <= 232448, "shared memory beyond the 227 KB a CTA may use");

struct Params {
    const uint8_t* q_sf;
    const uint8_t* k_sf;
    const uint8_t* v_sf;
    __nv_bfloat16* o;
    uint8_t* rollback_bits;
    unsigned long long* rollback_count;
    unsigned int* err_word;
    int S, D, n_t;
    float sm_scale;  // s = sm_scale * accumulator
    float alpha;     // 128 * log2(e) * sm_scale
    float theta;     // gate threshold, natural-log score units
    int p_off;       // 0: P in E4M3; 6: P on the E2M3 grid
    int p_emax;      // largest exponent of the P element type
    uint32_t p_mthr; // its largest mantissa in bf16 units
    uint64_t timeout_ns;
    int debug_flags;
};

__device__ __forceinline__ void raise_abort(Smem& sm, const Params& p) {
    sm.abort = 1;
    atomicOr(p.err_word, kErrTimeout);
}

// Smallest X with amax <= max_elem * 2^X, from the bf16 pattern of amax.
__device__ __forceinline__ int p_scale_exp(uint32_t amax_bf16, int emax, uint32_t mthr) {
    if (amax_bf16 == 0) return -127;
    int E = static_cast<int>(amax_bf16 >> 7);
    uint32_t m = amax_bf16 & 0x7Fu;
    int e;
    if (E == 0) {
        int nb = 32 - __clz(m);
        e = nb - 134;
        m = (m << (8 - nb)) & 0x7Fu;
    } else {
        e = E - 127;
    }
    int X = e - emax + (m > mthr ? 1 : 0);
    return min(127, max(-127, X));
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

// Max and min of 32 raw scores.
__device__ __forceinline__ void maxmin32(const uint32_t (&v)[32], float& mx, float& mn) {
    float a = fmax3(__uint_as_float(v[0]), __uint_as_float(v[1]), __uint_as_float(v[2]));
    float b = fmin3(__uint_as_float(v[0]), __uint_as_float(v[1]), __uint_as_float(v[2]));
#pragma unroll
    for (int j = 3; j < 31; j += 2) {
        a = fmax3(a, __uint_as_float(v[j]), __uint_as_float(v[j + 1]));
        b = fmin3(b, __uint_as_float(v[j]), __uint_as_float(v[j + 1]));
    }
    mx = fmaxf(a, __uint_as_float(v[31]));
    mn = fminf(b, __uint_as_float(v[31]));
}

// Keys at or beyond n_valid (relative to this 32-key chunk) become -inf.
__device__ __forceinline__ void mask32(uint32_t (&v)[32], int n_valid) {
#pragma unroll
    for (int j = 0; j < 32; ++j)
        if (j >= n_valid) v[j] = 0xFF800000u;
}

// Schraudolph code of a single score: rne(max(alpha * s + beta, 0)).  The
// upper clamp at 0x7F7F is never active: a row's scores never pass its
// reference by more than theta <= 80, so y <= 128 * (127 + 80 log2 e) - 7.
__device__ __forceinline__ uint32_t code_of(float s, float alpha, float beta) {
    const float y = fmaxf(__fmaf_rn(s, alpha, beta), 0.0f);
    return __float_as_uint(__fadd_rn(y, kMagic)) & 0xFFFFu;
}

// Two-stage conversion of 32 scores of one 32-key block: bf16 weight code
// (integer reinterpretation) -> E4M3 pattern of p * inv, inv = 2^-(X+off).
// Writes 8 words, element i in byte i % 4 of word i / 4.
template <bool kClamp>
__device__ __forceinline__ void convert32(const uint32_t (&v)[32], float alpha, float beta,
                                          float inv, uint32_t (&w)[8]) {
    const float2 a2 = make_float2(alpha, alpha), b2 = make_float2(beta, beta);
    const float2 m2 = make_float2(kMagic, kMagic), i2 = make_float2(inv, inv);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        float2 y = __ffma2_rn(make_float2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])),
                              a2, b2);
        if (kClamp) {
            y.x = fmaxf(y.x, 0.0f);
            y.y = fmaxf(y.y, 0.0f);
        }
        y = __fadd2_rn(y, m2);
        const float2 pw = make_float2(__uint_as_float(__float_as_uint(y.x) << 16),
                                      __uint_as_float(__float_as_uint(y.y) << 16));
        const float2 q = __fmul2_rn(pw, i2);
        const uint32_t e = cvt_e4m3x2(q.x, q.y);
        if (i & 1)
            w[i >> 1] |= e << 16;
        else
            w[i >> 1] = e;
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
// quotient to nearest even; its low byte is the E4M3 code.
__device__ __forceinline__ void convert32_linear(const uint32_t (&v)[32], float alpha, float beta,
                                                 float kx, uint32_t (&w)[8]) {
    const float2 a2 = make_float2(alpha, alpha), b2 = make_float2(beta, beta);
    const float2 m2 = make_float2(kMagic, kMagic), k2 = make_float2(kx, kx);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float2 y0 = __ffma2_rn(make_float2(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1])), a2, b2);
        float2 y1 = __ffma2_rn(make_float2(__uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3])), a2, b2);
        y0 = __fadd2_rn(__fadd2_rn(y0, m2), k2);
        y1 = __fadd2_rn(__fadd2_rn(y1, m2), k2);
        const uint32_t lo = __byte_perm(__float_as_uint(y0.x), __float_as_uint(y0.y), 0x0040);
        const uint32_t hi = __byte_perm(__float_as_uint(y1.x), __float_as_uint(y1.y), 0x0040);
        w[i] = __byte_perm(lo, hi, 0x5410);
    }
}

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
        mbar_init(&sm.bar_q, 1);
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&sm.kv_full[i], 1);
            mbar_init(&sm.kv_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.s_full[i], 1);
            mbar_init(&sm.s_free[i], 128);
            mbar_init(&sm.p_full[i], 128);
            mbar_init(&sm.p_free[i], 1);
            mbar_init(&sm.m_ready[i], 128);
        }
        mbar_init(&sm.o_full, 1);
        mbar_init(&sm.drain, 1);
        fence_mbar_init();
    }
    if (tid < 128) {
        // all-ones B operand (E4M3 1.0 = 0x38) and unit scales (2^0 = 127)
        reinterpret_cast<uint4*>(sm.ones)[tid] = make_uint4(0x38383838u, 0x38383838u, 0x38383838u, 0x38383838u);
        reinterpret_cast<uint32_t*>(sm.ones_sf)[tid] = 0x7F7F7F7Fu;
        fence_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;

    if (warp == kWarpLoad) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            const uint32_t tile_bytes = static_cast<uint32_t>(kTile * D);
            mbar_arrive_expect_tx(&sm.bar_q, tile_bytes + kAtomBytes);
            tma_load_3d(sm.q, &tm_q, &sm.bar_q, 0, q0, bh);
            bulk_load(sm.q_sf, p.q_sf + (static_cast<int64_t>(bh) * n_qt + qt) * kAtomBytes,
                      kAtomBytes, &sm.bar_q);
            int issued = 0;
            bool ok = true;
            for (int t = 0; t < p.n_t; ++t) {
                const int st = t % kStages;
                if (t >= kStages) {
                    if (!mbar_wait(&sm.kv_empty[st], ((t / kStages) - 1) & 1, p.timeout_ns,
                                   &sm.abort)) {
                        ok = false;
                        break;
                    }
                }
                if ((p.debug_flags & 1) && t == 1) continue;  // test: tile 1 never arrives
                mbar_arrive_expect_tx(&sm.kv_full[st], 2 * tile_bytes + 2 * kAtomBytes);
                tma_load_3d(sm.k[st], &tm_k, &sm.kv_full[st], 0, t * kTile, bh);
                tma_load_3d(sm.v[st], &tm_v, &sm.kv_full[st], t * kTile, 0, bh);
                const int64_t a = (static_cast<int64_t>(bh) * p.n_t + t) * kAtomBytes;
                bulk_load(sm.k_sf[st], p.k_sf + a, kAtomBytes, &sm.kv_full[st]);
                bulk_load(sm.v_sf[st], p.v_sf + a, kAtomBytes, &sm.kv_full[st]);
                issued = t + 1;
            }
            if (!ok) raise_abort(sm, p);
            if (sm.abort) {
                // let the copies still in flight land before the CTA exits
                int dummy = 0;
                mbar_wait(&sm.bar_q, 0, p.timeout_ns, &dummy);
                for (int t = max(0, issued - kStages); t < issued; ++t) {
                    if ((p.debug_flags & 1) && t == 1) continue;
                    mbar_wait(&sm.kv_full[t % kStages], (t / kStages) & 1, p.timeout_ns, &dummy);
                }
            }
        }
    } else if (warp == kWarpMma) {
        // ---------------------------------------------------------- MMA
        if (lane == 0) {
            const uint32_t idesc_qk0 = idesc_mxf8f6f4(128, 128, 0, 0, 0, 0);
            const uint32_t idesc_pv0 = idesc_mxf8f6f4(128, D, 0, 0, 0, 0);
            const uint32_t idesc_l0 = idesc_mxf8f6f4(128, 16, 0, 0, 0, 0);
            const uint32_t qk_swz = D == 128 ? SWZ_128B : SWZ_64B;
            const uint32_t qk_sbo = D == 128 ? 1024u : 512u;
            bool ok = mbar_wait(&sm.bar_q, 0, p.timeout_ns, &sm.abort);
            if (ok) {
                tc_fence_after();
                tc_cp_32x128b_x4(tmem + kColSfQ, smem_desc(smem_u32(sm.q_sf), 0, 128, SWZ_NONE));
                tc_cp_32x128b_x4(tmem + kColSfOnes, smem_desc(smem_u32(sm.ones_sf), 0, 128, SWZ_NONE));
            }
            auto issue_pv = [&](int u) {
                const int pb = u & 1, st = u % kStages;
                tc_fence_after();
                tc_cp_32x128b_x4(tmem + kColSfP + 4 * pb, smem_desc(smem_u32(sm.p_sf[pb]), 0, 128, SWZ_NONE));
                tc_cp_32x128b_x4(tmem + kColSfV + 4 * pb, smem_desc(smem_u32(sm.v_sf[st]), 0, 128, SWZ_NONE));
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint32_t sf = static_cast<uint32_t>(kk);
                    const uint64_t ad = smem_desc(smem_u32(sm.p[pb]) + 32 * kk, 16, 1024, SWZ_128B);
                    const uint64_t bd = smem_desc(smem_u32(sm.v[st]) + 32 * kk, 16, 1024, SWZ_128B);
                    mma_mxf8f6f4(tmem + kColO, ad, bd, idesc_pv0 | (sf << 4) | (sf << 29),
                                 tmem + kColSfP + 4 * pb, tmem + kColSfV + 4 * pb,
                                 (u > 0 || kk > 0) ? 1u : 0u);
                }
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint32_t sf = static_cast<uint32_t>(kk);
                    const uint64_t ad = smem_desc(smem_u32(sm.p[pb]) + 32 * kk, 16, 1024, SWZ_128B);
                    const uint64_t bd = smem_desc(smem_u32(sm.ones) + 32 * kk, 16, 1024, SWZ_128B);
                    mma_mxf8f6f4(tmem + kColL, ad, bd, idesc_l0 | (sf << 4) | (sf << 29),
                                 tmem + kColSfP + 4 * pb, tmem + kColSfOnes,
                                 (u > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(&sm.kv_empty[st]);
                tc_commit(&sm.p_free[pb]);
            };
            // Issue order: a score product as soon as its K tile landed and its
            // S buffer was released, ahead of any pending PV, so that a softmax
            // warpgroup never waits behind the other warpgroup's P.  Each
            // barrier below cannot complete its next phase before this thread
            // issues the corresponding MMA, so the parities are unambiguous.
            int qk = 0, pv = 0;
            uint64_t idle_since = globaltimer_ns();
            while (ok && pv < p.n_t) {
                bool progressed = false;
                if (qk < p.n_t) {
                    const int st = qk % kStages, sb = qk & 1;
                    if (mbar_test(&sm.kv_full[st], (qk / kStages) & 1) &&
                        (qk < 2 || mbar_test(&sm.s_free[sb], ((qk - 2) >> 1) & 1))) {
                        tc_fence_after();
                        tc_cp_32x128b_x4(tmem + kColSfK + 4 * sb, smem_desc(smem_u32(sm.k_sf[st]), 0, 128, SWZ_NONE));
                        for (int kk = 0; kk < nkk; ++kk) {
                            const uint32_t sf = static_cast<uint32_t>(kk);
                            const uint64_t ad = smem_desc(smem_u32(sm.q) + 32 * kk, 16, qk_sbo, qk_swz);
                            const uint64_t bd = smem_desc(smem_u32(sm.k[st]) + 32 * kk, 16, qk_sbo, qk_swz);
                            mma_mxf8f6f4(tmem + kColS0 + 128 * sb, ad, bd,
                                         idesc_qk0 | (sf << 4) | (sf << 29), tmem + kColSfQ,
                                         tmem + kColSfK + 4 * sb, kk > 0 ? 1u : 0u);
                        }
                        tc_commit(&sm.s_full[sb]);
                        ++qk;
                        progressed = true;
                    }
                }
                if (!progressed && pv < qk && mbar_test(&sm.p_full[pv & 1], (pv >> 1) & 1)) {
                    issue_pv(pv);
                    ++pv;
                    progressed = true;
                }
                if (progressed) {
                    idle_since = globaltimer_ns();
                } else if (sm.abort || globaltimer_ns() - idle_since > p.timeout_ns) {
                    ok = false;
                } else {
                    __nanosleep(32);  // leave the issue slots to the softmax warps
                }
            }
            if (ok) tc_commit(&sm.o_full);
            if (!ok) {
                raise_abort(sm, p);
                int dummy = 0;
                tc_commit(&sm.drain);  // wait until every issued MMA/copy retired
                mbar_wait(&sm.drain, 0, p.timeout_ns, &dummy);
            }
        }
    } else {
        // ------------------------------------------------------ softmax
        // Warpgroup wg processes the KV tiles t = wg, wg + 2, ... in TMEM S
        // buffer wg and shared P buffer wg; thread r owns query row r (TMEM
        // lane r).  The reference maximum travels between the warpgroups
        // through m_ref / m_ready after every tile.
        const int wg = warp >> 2;
        const int r = tid & 127;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        const uint32_t s_col = lane_addr + kColS0 + 128 * wg;
        const bool row_valid = (q0 + r) < p.S;
        const int64_t grow = static_cast<int64_t>(bh) * p.S + q0 + r;
        uint8_t* const prow = sm.p[wg] + (r >> 3) * 1024 + (r & 7) * 128;
        float m_acc = 0.0f;  // reference maximum in accumulator units
        unsigned fired_total = 0;
        bool ok = true;
        auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
            const bool w = mbar_wait(bar, parity, p.timeout_ns, &sm.abort);
            return __all_sync(0xFFFFFFFFu, w);
        };
        for (int t = wg, it = 0; t < p.n_t; t += 2, ++it) {
            if (!wait_all(&sm.s_full[wg], it & 1)) { ok = false; break; }
            tc_fence_after();
            const int n_valid = min(kTile, p.S - t * kTile);
            const bool tail = n_valid < kTile;
            // pass 1: block maxima and minima of the raw scores
            float bmax[4], bmin[4];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t v0[32], v1[32];
                tmem_ld32(s_col + 64 * h, v0);
                tmem_ld32(s_col + 64 * h + 32, v1);
                tmem_ld_wait();
                if (tail) {
                    mask32(v0, n_valid - 64 * h);
                    mask32(v1, n_valid - 64 * h - 32);
                }
                maxmin32(v0, bmax[2 * h], bmin[2 * h]);
                maxmin32(v1, bmax[2 * h + 1], bmin[2 * h + 1]);
            }
            const float tmax = fmaxf(fmaxf(bmax[0], bmax[1]), fmaxf(bmax[2], bmax[3]));
            // frozen reference: tile 0 sets it, the previous tile hands it on
            if (t > 0) {
                if (!wait_all(&sm.m_ready[wg ^ 1], ((t - 1) >> 1) & 1)) { ok = false; break; }
                m_acc = sm.m_ref[wg ^ 1][r];
            }
            bool fire = false;
            float rescale = 1.0f;
            if (t == 0) {
                m_acc = tmax;
            } else if ((tmax - m_acc) * p.sm_scale > p.theta) {
                fire = true;
                rescale = expf((m_acc - tmax) * p.sm_scale);
                m_acc = tmax;
            }
            sm.m_ref[wg][r] = m_acc;
            mbar_arrive(&sm.m_ready[wg]);
            if (p.rollback_bits && row_valid) p.rollback_bits[grow * p.n_t + t] = fire ? 1 : 0;
            fired_total += (fire && row_valid) ? 1u : 0u;
            const bool any_fire = __any_sync(0xFFFFFFFFu, fire);
            if (any_fire) {
                // recovery: once PV of the previous tile retired, O and l of the
                // firing rows are scaled by exp(m_old - m_new) in TMEM
                if (!wait_all(&sm.p_free[wg ^ 1], ((t - 1) >> 1) & 1)) { ok = false; break; }
                tc_fence_after();
                uint32_t rr[32];
                for (int c = 0; c < D / 32; ++c) {
                    tmem_ld32(lane_addr + kColO + 32 * c, rr);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) rr[j] = __float_as_uint(__uint_as_float(rr[j]) * rescale);
                    tmem_st32(lane_addr + kColO + 32 * c, rr);
                }
                uint32_t lv;
                tmem_ld1(lane_addr + kColL, lv);
                tmem_ld_wait();
                tmem_st1(lane_addr + kColL, __float_as_uint(__uint_as_float(lv) * rescale));
                tmem_st_wait();
            }
            // P buffer wg is free once PV of tile t - 2 retired
            if (t >= 2 && !wait_all(&sm.p_free[wg], (it - 1) & 1)) { ok = false; break; }
            const float beta = 16249.0f - p.alpha * m_acc;
            // pass 2: per 32-key block, E8M0 scale from the block's largest
            // weight code, then the conversion of its 32 scores
            uint32_t sfw = 0;
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                uint32_t v0[32], v1[32];
                tmem_ld32(s_col + 64 * h, v0);
                tmem_ld32(s_col + 64 * h + 32, v1);
                tmem_ld_wait();
                if (h == 1) {
                    // the whole S tile has been read: release the buffer so the
                    // next score product can start while this half converts
                    tc_fence_before();
                    mbar_arrive(&sm.s_free[wg]);
                }
                if (tail) {
                    mask32(v0, n_valid - 64 * h);
                    mask32(v1, n_valid - 64 * h - 32);
                }
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int b = 2 * h + e;
                    const float bx = h ? (e ? bmax[3] : bmax[2]) : (e ? bmax[1] : bmax[0]);
                    const float bn = h ? (e ? bmin[3] : bmin[2]) : (e ? bmin[1] : bmin[0]);
                    const int X = p_scale_exp(code_of(bx, p.alpha, beta), p.p_emax, p.p_mthr) + p.p_off;
                    const float inv = __int_as_float((127 - X) << 23);
                    sfw |= static_cast<uint32_t>(X + 127) << (8 * b);
                    uint32_t w[8];
                    // E4M3 P: the whole block converts to E4M3 normals when its
                    // smallest code is a normal bf16 (>= 128) and at least
                    // 128 X + 15488 (p / 2^X >= 2^-6)
                    const bool linear = p.p_off == 0 &&
                        __all_sync(0xFFFFFFFFu, static_cast<int>(code_of(bn, p.alpha, beta)) >= max(128, 128 * X + 15488));
                    if (linear) {
                        convert32_linear(e ? v1 : v0, p.alpha, beta,
                                         static_cast<float>(188728320 - 128 * X), w);
                    } else if (__any_sync(0xFFFFFFFFu, __fmaf_rn(bn, p.alpha, beta) < 0.0f)) {
                        convert32<true>(e ? v1 : v0, p.alpha, beta, inv, w);
                    } else {
                        convert32<false>(e ? v1 : v0, p.alpha, beta, inv, w);
                    }
                    *reinterpret_cast<uint4*>(prow + (((2 * b) ^ (r & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
                    *reinterpret_cast<uint4*>(prow + (((2 * b + 1) ^ (r & 7)) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
                }
            }
            tc_fence_before();
            *reinterpret_cast<uint32_t*>(sm.p_sf[wg] + (r & 31) * 16 + (r >> 5) * 4) = sfw;
            fence_async_smem();
            mbar_arrive(&sm.p_full[wg]);
        }
        if (!ok) raise_abort(sm, p);
        if (ok) {
            ok = wait_all(&sm.o_full, 0);
            if (!ok) raise_abort(sm, p);
        }
        if (ok) {
            // epilogue: warpgroup wg writes columns [wg * D/2, (wg+1) * D/2)
            tc_fence_after();
            uint32_t lv;
            tmem_ld1(lane_addr + kColL, lv);
            tmem_ld_wait();
            const float l = __uint_as_float(lv);
            for (int c = wg * (D / 64); c < (wg + 1) * (D / 64); ++c) {
                uint32_t rr[32];
                tmem_ld32(lane_addr + kColO + 32 * c, rr);
                tmem_ld_wait();
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
            if (p.rollback_count) {
                unsigned tot = fired_total;
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

}  // namespace

cudaError_t launch_fsa_attention(const AttnLaunch& a, cudaStream_t st) {
    Params p{};
    p.q_sf = a.ws.qsf;
    p.k_sf = a.ws.ksf;
    p.v_sf = a.ws.vsf;
    p.o = reinterpret_cast<__nv_bfloat16*>(a.o);
    p.rollback_bits = a.rollback_bits;
    p.rollback_count = a.rollback_count;
    p.err_word = a.err_word;
    p.S = a.S;
    p.D = a.D;
    p.n_t = (a.S + kTile - 1) / kTile;
    p.sm_scale = a.sm_scale;
    p.alpha = static_cast<float>(128.0 * 1.4426950408889634 * static_cast<double>(a.sm_scale));
    p.theta = a.threshold;
    const bool p_e4m3 = (a.fmt == 0);
    p.p_off = p_e4m3 ? 0 : 6;
    p.p_emax = p_e4m3 ? 8 : 2;
    p.p_mthr = p_e4m3 ? 0x60u : 0x70u;
    p.timeout_ns = a.timeout_ns;
    p.debug_flags = a.debug_flags;
    const size_t smem = sizeof(Smem);
    cudaError_t e = cudaFuncSetAttribute(fsa_attn_fwd_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    dim3 grid(static_cast<unsigned>(p.n_t), static_cast<unsigned>(a.BH));
    fsa_attn_fwd_kernel<<<grid, kThreads, smem, st>>>(*a.tm_q, *a.tm_k, *a.tm_v, p);
    return cudaGetLastError();
}

}  // namespace fsa
