// bf16_attention.cu -- conventional BF16 flash attention for sm_103a: the
// speed and error denominator of the quantized kernel ("Fused-Softmax shifts
// an AI attention bottleneck onto faster GPU hardware", paragraphs 7-8 compare
// against BF16 attention).
//
// Exact softmax with a running row maximum: p = exp2((s - m) * sm * log2 e)
// with the CUDA exp2f, P rounded to bf16, O += P V on tcgen05 kind::f16 with
// FP32 accumulation in TMEM, l summed in FP32 on the CUDA cores, O and l
// rescaled by exp2(m_old - m_new) whenever a row's maximum grows.
//
// Same decomposition as the MX kernel: one CTA per (128-row query tile,
// head); two softmax warpgroups take alternate KV tiles (thread = row = TMEM
// lane), warp 8 is the TMA producer, warp 9 the TMEM allocator + MMA issuer.  Q and K are K-major (128-byte
// swizzle, 64 bf16 per swizzle row); V is read in its natural [keys][D]
// layout as an MN-major B operand.
#include <cuda_bf16.h>

#include "fsa_internal.h"
#include "sm100_ptx.cuh"

namespace fsa {
namespace {

constexpr int kStages = 2;
constexpr int kThreads = 320;          // 2 softmax warpgroups + loader warp + MMA warp
constexpr int kWarpLoad = 8, kWarpMma = 9;
constexpr int kAtom = 128 * 128;         // 128 rows x 128 bytes (64 bf16)
constexpr int kTileBytes = 2 * kAtom;    // 128 rows x 128 bf16
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS0 = 0, kColO = 256;  // S1 = kColS0 + 128

struct __align__(1024) Smem {
    uint8_t q[kTileBytes];
    uint8_t k[kStages][kTileBytes];
    uint8_t v[kStages][kTileBytes];
    uint8_t p[2][kTileBytes];
    float m_run[2][128];   // running maximum handed between the warpgroups
    float l_part[2][128];  // each warpgroup's final partial row sum (relative to m_run)
    uint64_t bar_q;
    uint64_t kv_full[kStages];
    uint64_t kv_empty[kStages];
    uint64_t s_full[2];
    uint64_t s_free[2];
    uint64_t p_full[2];
    uint64_t p_free[2];
    uint64_t m_ready[2];
    uint64_t fin_ready;
    uint64_t o_full;
    uint64_t drain;
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

__device__ __forceinline__ float max32(const uint32_t (&v)[32]) {
    float a = fmax3(__uint_as_float(v[0]), __uint_as_float(v[1]), __uint_as_float(v[2]));
#pragma unroll
    for (int j = 3; j < 31; j += 2) a = fmax3(a, __uint_as_float(v[j]), __uint_as_float(v[j + 1]));
    return fmaxf(a, __uint_as_float(v[31]));
}

__device__ __forceinline__ void mask32(uint32_t (&v)[32], int n_valid) {
#pragma unroll
    for (int j = 0; j < 32; ++j)
        if (j >= n_valid) v[j] = 0xFF800000u;
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
        mbar_init(&sm.fin_ready, 256);
        for (int i = 0; i < 256; ++i) {
            (&sm.m_run[0][0])[i] = -INFINITY;
            (&sm.l_part[0][0])[i] = 0.0f;
        }
        mbar_init(&sm.o_full, 1);
        mbar_init(&sm.drain, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;

    if (warp == kWarpLoad) {
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            const uint32_t atom_bytes = static_cast<uint32_t>(kTile * 128);
            mbar_arrive_expect_tx(&sm.bar_q, atom_bytes * n_atoms);
            for (int a = 0; a < n_atoms; ++a) tma_load_3d(sm.q + a * kAtom, &tm_q, &sm.bar_q, 64 * a, q0, bh);
            int issued = 0;
            bool ok = true;
            for (int t = 0; t < p.n_t; ++t) {
                const int st = t % kStages;
                if (t >= kStages &&
                    !mbar_wait(&sm.kv_empty[st], ((t / kStages) - 1) & 1, p.timeout_ns, &sm.abort)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&sm.kv_full[st], 2 * atom_bytes * n_atoms);
                for (int a = 0; a < n_atoms; ++a) {
                    tma_load_3d(sm.k[st] + a * kAtom, &tm_k, &sm.kv_full[st], 64 * a, t * kTile, bh);
                    tma_load_3d(sm.v[st] + a * kAtom, &tm_v, &sm.kv_full[st], 64 * a, t * kTile, bh);
                }
                issued = t + 1;
            }
            if (!ok) raise_abort(sm, p);
            if (sm.abort) {
                int dummy = 0;
                mbar_wait(&sm.bar_q, 0, p.timeout_ns, &dummy);
                for (int t = max(0, issued - kStages); t < issued; ++t)
                    mbar_wait(&sm.kv_full[t % kStages], (t / kStages) & 1, p.timeout_ns, &dummy);
            }
        }
    } else if (warp == kWarpMma) {
        if (lane == 0) {
            const uint32_t idesc_qk = idesc_bf16(128, 128, 0, 0);
            const uint32_t idesc_pv = idesc_bf16(128, D, 0, 1);
            bool ok = mbar_wait(&sm.bar_q, 0, p.timeout_ns, &sm.abort);
            auto issue_pv = [&](int u) -> bool {
                const int st = u % kStages, pb = u & 1;
                if (!mbar_wait(&sm.p_full[pb], (u >> 1) & 1, p.timeout_ns, &sm.abort)) return false;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {  // 16 keys per step
                    const uint64_t ad = smem_desc(smem_u32(sm.p[pb]) + (kk >> 2) * kAtom + 32 * (kk & 3), 16,
                                                  1024, SWZ_128B);
                    // V: MN-major; 64-wide d atoms kAtom apart (LBO), 8-key groups 1024 apart (SBO)
                    const uint64_t bd = smem_desc(smem_u32(sm.v[st]) + kk * 16 * 128, kAtom, 1024, SWZ_128B);
                    mma_bf16(tmem + kColO, ad, bd, idesc_pv, (u > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(&sm.kv_empty[st]);
                tc_commit(&sm.p_free[pb]);
                return true;
            };
            for (int t = 0; ok && t < p.n_t; ++t) {
                const int st = t % kStages, sb = t & 1;
                if (!mbar_wait(&sm.kv_full[st], (t / kStages) & 1, p.timeout_ns, &sm.abort)) { ok = false; break; }
                if (t >= 2 && !mbar_wait(&sm.s_free[sb], ((t - 2) >> 1) & 1, p.timeout_ns, &sm.abort)) { ok = false; break; }
                tc_fence_after();
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kAtom + 32 * (kk & 3);
                    const uint64_t ad = smem_desc(smem_u32(sm.q) + off, 16, 1024, SWZ_128B);
                    const uint64_t bd = smem_desc(smem_u32(sm.k[st]) + off, 16, 1024, SWZ_128B);
                    mma_bf16(tmem + kColS0 + 128 * sb, ad, bd, idesc_qk, kk > 0 ? 1u : 0u);
                }
                tc_commit(&sm.s_full[sb]);
                if (t >= 1 && !issue_pv(t - 1)) { ok = false; break; }
            }
            if (ok && !issue_pv(p.n_t - 1)) ok = false;
            if (ok) tc_commit(&sm.o_full);
            if (!ok) {
                raise_abort(sm, p);
                int dummy = 0;
                tc_commit(&sm.drain);
                mbar_wait(&sm.drain, 0, p.timeout_ns, &dummy);
            }
        }
    } else {
        // softmax warpgroup wg: KV tiles wg, wg + 2, ...; thread r = row r.
        // The running maximum is handed between the warpgroups after every
        // tile; each warpgroup keeps its own partial row sum relative to the
        // maximum of its latest tile, combined at the end.
        const int wg = warp >> 2;
        const int r = tid & 127;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        const uint32_t s_col = lane_addr + kColS0 + 128 * wg;
        const bool row_valid = (q0 + r) < p.S;
        const int64_t grow = static_cast<int64_t>(bh) * p.S + q0 + r;
        float m = -INFINITY;  // running max of s * c
        float l = 0.0f;       // this warpgroup's partial sum, relative to m
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
            float tmax = -INFINITY;
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
                tmax = fmax3(tmax, max32(v0), max32(v1));
            }
            float m_prev = m;
            if (t > 0) {
                if (!wait_all(&sm.m_ready[wg ^ 1], ((t - 1) >> 1) & 1)) { ok = false; break; }
                m_prev = sm.m_run[wg ^ 1][r];
            }
            const float m_new = fmaxf(m_prev, tmax * p.c);
            sm.m_run[wg][r] = m_new;
            mbar_arrive(&sm.m_ready[wg]);
            // O (all tiles so far) is relative to m_prev; rescale when it grew
            const bool grew = m_new > m_prev;
            if (t >= 1 && __any_sync(0xFFFFFFFFu, grew)) {
                if (!wait_all(&sm.p_free[wg ^ 1], ((t - 1) >> 1) & 1)) { ok = false; break; }
                tc_fence_after();
                const float corr = exp2f(m_prev - m_new);
                uint32_t rr[32];
                for (int c = 0; c < D / 32; ++c) {
                    tmem_ld32(lane_addr + kColO + 32 * c, rr);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) rr[j] = __float_as_uint(__uint_as_float(rr[j]) * corr);
                    tmem_st32(lane_addr + kColO + 32 * c, rr);
                }
                tmem_st_wait();
            }
            if (t >= 2 && !wait_all(&sm.p_free[wg], (it - 1) & 1)) { ok = false; break; }
            // own partial sum follows the new maximum
            l = (m == -INFINITY) ? 0.0f : l * exp2f(m - m_new);
            m = m_new;
            float ls = 0.0f;
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                uint32_t v0[32], v1[32];
                tmem_ld32(s_col + 64 * h, v0);
                tmem_ld32(s_col + 64 * h + 32, v1);
                tmem_ld_wait();
                if (tail) {
                    mask32(v0, n_valid - 64 * h);
                    mask32(v1, n_valid - 64 * h - 32);
                }
                uint8_t* prow = sm.p[wg] + h * kAtom + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    uint32_t pk[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const uint32_t* v = e ? v1 : v0;
                        const float a = exp2f(__fmaf_rn(__uint_as_float(v[2 * j]), p.c, -m));
                        const float b = exp2f(__fmaf_rn(__uint_as_float(v[2 * j + 1]), p.c, -m));
                        __nv_bfloat162 h2 = __floats2bfloat162_rn(a, b);
                        ls += __low2float(h2) + __high2float(h2);
                        pk[j] = *reinterpret_cast<uint32_t*>(&h2);
                    }
#pragma unroll
                    for (int ch = 0; ch < 4; ++ch) {
                        const int c = 4 * e + ch;  // 16-byte chunk within the 128-byte row
                        *reinterpret_cast<uint4*>(prow + ((c ^ (r & 7)) << 4)) =
                            make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
                    }
                }
            }
            l += ls;
            tc_fence_before();
            mbar_arrive(&sm.s_free[wg]);
            fence_async_smem();
            mbar_arrive(&sm.p_full[wg]);
        }
        if (!ok) raise_abort(sm, p);
        // combine the two partial sums: l = sum_w l_w * 2^(m_w - m_final)
        if (ok) {
            sm.l_part[wg][r] = l;
            mbar_arrive(&sm.fin_ready);
            ok = wait_all(&sm.fin_ready, 0);
            if (!ok) raise_abort(sm, p);
        }
        if (ok) {
            ok = wait_all(&sm.o_full, 0);
            if (!ok) raise_abort(sm, p);
        }
        if (ok) {
            const float m0 = sm.m_run[0][r], l0 = sm.l_part[0][r];
            const float m1 = sm.m_run[1][r], l1 = sm.l_part[1][r];
            const float mf = fmaxf(m0, m1);
            const float lt = (m0 == -INFINITY ? 0.0f : l0 * exp2f(m0 - mf)) +
                             (m1 == -INFINITY ? 0.0f : l1 * exp2f(m1 - mf));
            tc_fence_after();
            for (int c = wg * (D / 64); c < (wg + 1) * (D / 64); ++c) {
                uint32_t rr[32];
                tmem_ld32(lane_addr + kColO + 32 * c, rr);
                tmem_ld_wait();
                if (row_valid) {
                    uint32_t packed[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        __nv_bfloat162 h2 = __floats2bfloat162_rn(__fdiv_rn(__uint_as_float(rr[2 * j]), lt),
                                                                  __fdiv_rn(__uint_as_float(rr[2 * j + 1]), lt));
                        packed[j] = *reinterpret_cast<uint32_t*>(&h2);
                    }
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
    cudaError_t e = cudaFuncSetAttribute(bf16_attn_fwd_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    dim3 grid(static_cast<unsigned>(p.n_t), static_cast<unsigned>(a.BH));
    bf16_attn_fwd_kernel<<<grid, kThreads, smem, st>>>(*a.tm_q, *a.tm_k, *a.tm_v, p);
    return cudaGetLastError();
}

}  // namespace fsa
