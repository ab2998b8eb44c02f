// bf16_attention.cu -- conventional BF16 flash attention for sm_103a: the
// speed and error denominator of the quantized kernel ("Fused-Softmax shifts
// an AI attention bottleneck onto faster GPU hardware", paragraphs 7-8 compare
// against BF16 attention).
//
// Exact softmax with a running row maximum: p = 2^(s * sm * log2 e - m) with
// the hardware ex2 (SFU), P rounded to bf16, O += P V on tcgen05 kind::f16
// with FP32 accumulation in TMEM, l summed in FP32 on the CUDA cores, and O
// rescaled by 2^(m_old - m_new) whenever a row's maximum grows.
//
// Same machine as the MX kernel (the softmax is the conventional one): one
// CTA per (128-row query tile, head), 12 warps:
//   warps 0-3 / 4-7  softmax warpgroups 0 / 1: KV tiles 0, 2, ... / 1, 3, ...
//                    (thread = row = TMEM lane); the tile maxima are handed
//                    from one warpgroup to the other and each replays the
//                    running maximum over them;
//   warp 8           TMA producer of Q and the K ring; warp 10 of the V ring;
//   warp 9           TMEM allocator and issuer of the score products;
//   warp 11          issuer of the PV products, A = P read from TMEM.
// Q and K are K-major (128-byte swizzle, 64 bf16 per swizzle row); V is read
// in its natural [keys][D] layout as an MN-major B operand.
#include <cuda_bf16.h>

#include "fsa_internal.h"
#include "sm100_ptx.cuh"

namespace fsa {
namespace {

constexpr int kKStages = 3, kVStages = 2;
constexpr int kThreads = 384;
constexpr int kWarpLoad = 8, kWarpMma = 9, kWarpLoadV = 10, kWarpPv = 11;
// launched at 168 registers per thread; helpers drop to 32, softmax takes 232
constexpr int kLaunchRegs = 168, kSoftmaxRegs = 232, kHelperRegs = 32;
static_assert(2 * 128 * kSoftmaxRegs + 128 * kHelperRegs <= kThreads * kLaunchRegs,
              "register split exceeds the launch allocation");
constexpr int kAtom = 128 * 128;         // 128 rows x 128 bytes (64 bf16)
constexpr int kTileBytes = 2 * kAtom;    // 128 rows x 128 bf16
constexpr uint32_t kTmemCols = 512;
// TMEM columns: S0, S1 (128 each), O (D), P0, P1 (64 each: 128 bf16 per row)
constexpr uint32_t kColS0 = 0, kColO = 256, kColP = 384;

struct __align__(1024) Smem {
    uint8_t q[kTileBytes];
    uint8_t k[kKStages][kTileBytes];
    uint8_t v[kVStages][kTileBytes];
    float tmax_x[8][128];  // scaled row maxima of tile t in slot t % 8, read by the other warpgroup
    float l_fin[2][128];   // each warpgroup's final partial row sum (relative to m_fin)
    float m_fin[2][128];
    uint64_t bar_q;
    uint64_t k_full[kKStages], k_empty[kKStages];
    uint64_t v_full[kVStages], v_empty[kVStages];
    uint64_t s_full[2], s_free[2];
    uint64_t p_full[2], p_free[2];
    uint64_t m_ready[8];
    uint64_t fin_ready;
    uint64_t o_full;
    uint64_t drain_qk, drain_pv;
    uint32_t tmem_base;
    int abort;
};

static_assert(sizeof(Smem) <= 232448, "shared memory beyond the 227 KB a CTA may use");

struct Params {
    __nv_bfloat16* o;
    unsigned int* err_word;
    int S, D, n_t;
    float c;  // sm_scale * log2(e)
    uint64_t timeout_ns;
};

__device__ __forceinline__ void raise_abort(Smem& sm, const Params& p) {
    sm.abort = 1;
    atomicOr(p.err_word, kErrTimeout);
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// 2^x on the SFU (flushes results below 2^-126 to zero).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
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

__device__ __forceinline__ void mask32(uint32_t (&v)[32], int n_valid) {
#pragma unroll
    for (int j = 0; j < 32; ++j)
        if (j >= n_valid) v[j] = 0xFF800000u;
}

// p = 2^(s c - m) for 32 scores, packed to 16 bf16 pairs in w; returns their FP32 sum.
__device__ __forceinline__ float exp32(const uint32_t (&v)[32], float c, float m, uint32_t (&w)[16]) {
    const float2 c2 = make_float2(c, c), nm2 = make_float2(-m, -m);
    float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float2 x = __ffma2_rn(make_float2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])), c2, nm2);
        const float2 pp = make_float2(ex2(x.x), ex2(x.y));
        acc = __fadd2_rn(acc, pp);
        w[i] = bf16x2(pp.x, pp.y);
    }
    return acc.x + acc.y;
}

__device__ __forceinline__ void warp_arrive(uint64_t* bar) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// Per-row state of a softmax thread.
struct RowState {
    float m_run;  // running maximum (scaled) before the current tile, replayed
    float m_own;  // maximum this warpgroup's partial sum is relative to
    float l_own;  // this warpgroup's partial row sum
};

// One KV tile t (the it-th of warpgroup wg) for query row r: one TMEM read
// of the scores, the tile maximum handed to the other warpgroup, the running
// maximum, the O rescale when it grew, then P = 2^(s c - m) in bf16 into
// TMEM P buffer t % 2 and its FP32 sum into this warpgroup's partial l.
__device__ __forceinline__ bool softmax_tile(Smem& sm, const Params& p, int t, int it, int wg, int r,
                                             uint32_t lane_addr, uint32_t s_col, bool tail,
                                             RowState& rs) {
    const int D = p.D;
    const int pb = t & 1;
    bool ok = mbar_wait(&sm.s_full[wg], it & 1, p.timeout_ns, &sm.abort);
    tc_fence_after();
    uint32_t s0[32], s1[32], s2[32], s3[32];
    tmem_ld32(s_col, s0);
    tmem_ld32(s_col + 32, s1);
    tmem_ld32(s_col + 64, s2);
    tmem_ld32(s_col + 96, s3);
    // non-blocking looks at the other warpgroup's maximum of tile t - 1 and
    // at this tile's P buffer (PV of tile t - 2 retired) while the scores travel
    const int ms = (t - 1) & 7;
    const uint32_t m_par = ((t - 1) >> 3) & 1;
    const uint32_t pf_par = ((t >> 1) - 1) & 1;
    const bool have_prev = t == 0 || mbar_test(&sm.m_ready[ms], m_par);
    float prev = (t > 0 && have_prev) ? sm.tmax_x[ms][r] : 0.0f;
    const bool have_p = t < 2 || mbar_test(&sm.p_free[pb], pf_par);
    tmem_ld_wait();
    tmem_reg_dep(s0);
    tmem_reg_dep(s1);
    tmem_reg_dep(s2);
    tmem_reg_dep(s3);
    tc_fence_before();
    warp_arrive(&sm.s_free[wg]);
    if (tail) {
        const int n_valid = p.S - t * kTile;
        mask32(s0, n_valid);
        mask32(s1, n_valid - 32);
        mask32(s2, n_valid - 64);
        mask32(s3, n_valid - 96);
    }
    const float tmax = p.c * fmaxf(fmaxf(max32(s0), max32(s1)), fmaxf(max32(s2), max32(s3)));
    // the scaled tile maximum for the other warpgroup, slot t % 8
    sm.tmax_x[t & 7][r] = tmax;
    warp_arrive(&sm.m_ready[t & 7]);
    // running maximum before this tile: m_{t-1} = max(m_{t-2}, tmax_{t-1})
    if (t > 0) {
        if (!have_prev) {
            ok &= mbar_wait(&sm.m_ready[ms], m_par, p.timeout_ns, &sm.abort);
            prev = sm.tmax_x[ms][r];
        }
        rs.m_run = fmaxf(rs.m_run, prev);
    }
    const float m_new = fmaxf(rs.m_run, tmax);
    // P buffer pb is free once PV of tile t - 2 retired (waited first: PV
    // products retire in order, so tile t - 1's buffer is then in the phase
    // of PV_{t-1} itself)
    if (!have_p) ok &= mbar_wait(&sm.p_free[pb], pf_par, p.timeout_ns, &sm.abort);
    const bool grew = t > 0 && m_new > rs.m_run;
    if (__any_sync(0xFFFFFFFFu, grew)) {
        // O holds the tiles before t relative to m_{t-1}: once PV_{t-1}
        // retired, scale it to the new maximum
        ok &= mbar_wait(&sm.p_free[(t - 1) & 1], ((t - 1) >> 1) & 1, p.timeout_ns, &sm.abort);
        tc_fence_after();
        const float corr = ex2(rs.m_run - m_new);
        uint32_t rr[32];
        for (int c = 0; c < D / 32; ++c) {
            tmem_ld32(lane_addr + kColO + 32 * c, rr);
            tmem_ld_wait();
            tmem_reg_dep(rr);
#pragma unroll
            for (int j = 0; j < 32; ++j) rr[j] = __float_as_uint(__uint_as_float(rr[j]) * corr);
            tmem_st32(lane_addr + kColO + 32 * c, rr);
        }
        tmem_st_wait();
    }
    // this warpgroup's partial sum follows the new maximum
    rs.l_own = (rs.m_own == -INFINITY) ? 0.0f : rs.l_own * ex2(rs.m_own - m_new);
    rs.m_own = m_new;
    rs.m_run = m_new;
    uint32_t w0[16], w1[16], w2[16], w3[16];
    const float ls = (exp32(s0, p.c, m_new, w0) + exp32(s1, p.c, m_new, w1)) +
                     (exp32(s2, p.c, m_new, w2) + exp32(s3, p.c, m_new, w3));
    rs.l_own += ls;
    // the bf16 P row (64 columns) into TMEM, the A operand of the PV product
    uint32_t lo[32], hi[32];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        lo[j] = w0[j];
        lo[16 + j] = w1[j];
        hi[j] = w2[j];
        hi[16 + j] = w3[j];
    }
    tmem_st32(lane_addr + kColP + 64 * pb, lo);
    tmem_st32(lane_addr + kColP + 64 * pb + 32, hi);
    tmem_st_wait();
    tc_fence_before();
    warp_arrive(&sm.p_full[pb]);
    return __all_sync(0xFFFFFFFFu, ok);
}

__global__ void __launch_bounds__(kThreads, 1)
    bf16_attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const Params p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // the 128-byte-swizzled TMA/MMA tiles need a 1024-byte aligned base
    if (smem_u32(smem_raw) & 1023u) {
        if (threadIdx.x == 0) atomicOr(p.err_word, kErrMisaligned);
        return;
    }
    Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q0 = blockIdx.x * kTile, bh = blockIdx.y;
    const int D = p.D;
    const int n_atoms = D / 64;  // swizzle atoms along D

    if (warp == kWarpMma) {
        tmem_alloc(&sm.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        sm.abort = 0;
        mbar_init(&sm.bar_q, 1);
        for (int i = 0; i < kKStages; ++i) {
            mbar_init(&sm.k_full[i], 1);
            mbar_init(&sm.k_empty[i], 1);
        }
        for (int i = 0; i < kVStages; ++i) {
            mbar_init(&sm.v_full[i], 1);
            mbar_init(&sm.v_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.s_full[i], 1);
            mbar_init(&sm.s_free[i], 4);  // one arrival per softmax warp
            mbar_init(&sm.p_full[i], 4);
            mbar_init(&sm.p_free[i], 1);
        }
        for (int i = 0; i < 8; ++i) mbar_init(&sm.m_ready[i], 4);
        mbar_init(&sm.fin_ready, 8);
        mbar_init(&sm.o_full, 1);
        mbar_init(&sm.drain_qk, 1);
        mbar_init(&sm.drain_pv, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    const uint32_t atom_bytes = static_cast<uint32_t>(kTile * 128);

    if (warp == kWarpLoad || warp == kWarpLoadV) {
        warpgroup_reg_dec<kHelperRegs>();
        // warp 8: Q once, then the K ring; warp 10: the V ring
        if (lane == 0) {
            const bool is_k = warp == kWarpLoad;
            const int stages = is_k ? kKStages : kVStages;
            uint64_t* full = is_k ? sm.k_full : sm.v_full;
            uint64_t* empty = is_k ? sm.k_empty : sm.v_empty;
            const CUtensorMap* map = is_k ? &tm_k : &tm_v;
            tma_prefetch_desc(map);
            if (is_k) {
                tma_prefetch_desc(&tm_q);
                mbar_arrive_expect_tx(&sm.bar_q, atom_bytes * n_atoms);
                for (int a = 0; a < n_atoms; ++a)
                    tma_load_3d(sm.q + a * kAtom, &tm_q, &sm.bar_q, 64 * a, q0, bh);
            }
            int issued = 0, st = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int t = 0; t < p.n_t; ++t) {
                if (t >= stages && !mbar_wait(&empty[st], ph ^ 1u, p.timeout_ns, &sm.abort)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&full[st], atom_bytes * n_atoms);
                uint8_t* dst = is_k ? sm.k[st] : sm.v[st];
                for (int a = 0; a < n_atoms; ++a)
                    tma_load_3d(dst + a * kAtom, map, &full[st], 64 * a, t * kTile, bh);
                issued = t + 1;
                if (++st == stages) {
                    st = 0;
                    ph ^= 1u;
                }
            }
            if (!ok) raise_abort(sm, p);
            if (sm.abort) {
                // let the copies still in flight land before the CTA exits
                int dummy = 0;
                if (is_k) mbar_wait(&sm.bar_q, 0, p.timeout_ns, &dummy);
                for (int t = max(0, issued - stages); t < issued; ++t)
                    mbar_wait(&full[t % stages], (t / stages) & 1, p.timeout_ns, &dummy);
            }
        }
    } else if (warp == kWarpMma || warp == kWarpPv) {
        warpgroup_reg_dec<kHelperRegs>();
        // Two issuing threads with descriptors built once: the start-address
        // field counts 16-byte units, so + 2 advances a K-major operand by one
        // 16-element K step and + kAtom / 16 by one swizzle atom.
        if (lane == 0) {
            bool ok = true;
            if (warp == kWarpMma) {
                const uint32_t id_qk = idesc_bf16(128, 128, 0, 0);
                const uint64_t dq = smem_desc(smem_u32(sm.q), 16, 1024, SWZ_128B);
                const uint64_t dk0 = smem_desc(smem_u32(sm.k[0]), 16, 1024, SWZ_128B);
                ok = mbar_wait(&sm.bar_q, 0, p.timeout_ns, &sm.abort);
                int st = 0;
                uint32_t ph = 0;
                for (int t = 0; ok && t < p.n_t; ++t) {
                    const int sb = t & 1;
                    if (t >= 2 && !mbar_wait(&sm.s_free[sb], ((t - 2) >> 1) & 1, p.timeout_ns, &sm.abort)) {
                        ok = false;
                        break;
                    }
                    if (!mbar_wait(&sm.k_full[st], ph, p.timeout_ns, &sm.abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t bk = dk0 + (kTileBytes >> 4) * st;
                    const uint32_t dst = tmem + kColS0 + 128 * sb;
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * (kAtom >> 4) + 2 * (kk & 3);
                        mma_bf16(dst, dq + off, bk + off, id_qk, kk > 0 ? 1u : 0u);
                    }
                    tc_commit(&sm.s_full[sb]);
                    tc_commit(&sm.k_empty[st]);
                    if (++st == kKStages) {
                        st = 0;
                        ph ^= 1u;
                    }
                }
            } else {
                // V MN-major: 64-wide d atoms kAtom apart (LBO), 8-key groups
                // 1024 apart (SBO); one 16-key K step is 2048 bytes
                const uint32_t id_pv = idesc_bf16(128, D, 0, 1);
                const uint64_t dv0 = smem_desc(smem_u32(sm.v[0]), kAtom, 1024, SWZ_128B);
                int st = 0;
                uint32_t ph = 0;
                for (int u = 0; ok && u < p.n_t; ++u) {
                    const int pb = u & 1;
                    if (!mbar_wait(&sm.p_full[pb], (u >> 1) & 1, p.timeout_ns, &sm.abort) ||
                        !mbar_wait(&sm.v_full[st], ph, p.timeout_ns, &sm.abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t ap = tmem + kColP + 64 * pb;  // 8 columns per 16-key step
                    const uint64_t bv = dv0 + (kTileBytes >> 4) * st;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_bf16_tmem_a(tmem + kColO, ap + 8 * kk, bv + 128 * kk, id_pv,
                                        (u > 0 || kk > 0) ? 1u : 0u);
                    tc_commit(&sm.v_empty[st]);
                    tc_commit(&sm.p_free[pb]);
                    if (++st == kVStages) {
                        st = 0;
                        ph ^= 1u;
                    }
                }
                if (ok) tc_commit(&sm.o_full);
            }
            if (!ok) {
                raise_abort(sm, p);
                int dummy = 0;
                uint64_t* drain = warp == kWarpMma ? &sm.drain_qk : &sm.drain_pv;
                tc_commit(drain);  // wait until every MMA this thread issued retired
                mbar_wait(drain, 0, p.timeout_ns, &dummy);
            }
        }
    } else {
        warpgroup_reg_inc<kSoftmaxRegs>();
        const int wg = warp >> 2;
        const int r = tid & 127;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        const uint32_t s_col = lane_addr + kColS0 + 128 * wg;
        const bool row_valid = (q0 + r) < p.S;
        const int64_t grow = static_cast<int64_t>(bh) * p.S + q0 + r;
        RowState rs{-INFINITY, -INFINITY, 0.0f};
        bool ok = true;
        const int t_tail = (p.S % kTile) ? p.n_t - 1 : p.n_t;
        for (int t = wg, it = 0; ok && t < p.n_t; t += 2, ++it)
            ok = softmax_tile(sm, p, t, it, wg, r, lane_addr, s_col, t == t_tail, rs);
        if (!ok) raise_abort(sm, p);
        // combine the two partial sums: l = sum_w l_w * 2^(m_w - m_final)
        if (ok) {
            sm.l_fin[wg][r] = rs.l_own;
            sm.m_fin[wg][r] = rs.m_own;
            warp_arrive(&sm.fin_ready);
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(&sm.fin_ready, 0, p.timeout_ns, &sm.abort));
            if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait(&sm.o_full, 0, p.timeout_ns, &sm.abort));
            if (!ok) raise_abort(sm, p);
        }
        if (ok) {
            const float m0 = sm.m_fin[0][r], l0 = sm.l_fin[0][r];
            const float m1 = sm.m_fin[1][r], l1 = sm.l_fin[1][r];
            const float mf = fmaxf(m0, m1);
            const float lt = (m0 == -INFINITY ? 0.0f : l0 * ex2(m0 - mf)) +
                             (m1 == -INFINITY ? 0.0f : l1 * ex2(m1 - mf));
            tc_fence_after();
            for (int c = wg * (D / 64); c < (wg + 1) * (D / 64); ++c) {
                uint32_t rr[32];
                tmem_ld32(lane_addr + kColO + 32 * c, rr);
                tmem_ld_wait();
                tmem_reg_dep(rr);
                if (row_valid) {
                    uint32_t packed[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        packed[j] = bf16x2(__fdiv_rn(__uint_as_float(rr[2 * j]), lt),
                                           __fdiv_rn(__uint_as_float(rr[2 * j + 1]), lt));
                    uint4* dst = reinterpret_cast<uint4*>(p.o + grow * D + 32 * c);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        dst[j] = make_uint4(packed[4 * j], packed[4 * j + 1], packed[4 * j + 2], packed[4 * j + 3]);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

cudaError_t launch_bf16_attention(const Bf16Launch& a, cudaStream_t st) {
    Params p{};
    p.o = reinterpret_cast<__nv_bfloat16*>(a.o);
    p.err_word = a.err_word;
    p.S = a.S;
    p.D = a.D;
    p.n_t = (a.S + kTile - 1) / kTile;
    p.c = static_cast<float>(static_cast<double>(a.sm_scale) * 1.4426950408889634);
    p.timeout_ns = a.timeout_ns;
    const size_t smem = sizeof(Smem);
    // the in-kernel register split assumes exactly kLaunchRegs per thread at
    // launch; anything else could make the increase wait forever
    cudaFuncAttributes fa{};
    cudaError_t e = cudaFuncGetAttributes(&fa, bf16_attn_fwd_kernel);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(bf16_attn_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    dim3 grid(static_cast<unsigned>(p.n_t), static_cast<unsigned>(a.BH));
    bf16_attn_fwd_kernel<<<grid, kThreads, smem, st>>>(*a.tm_q, *a.tm_k, *a.tm_v, p);
    return cudaGetLastError();
}

}  // namespace fsa
