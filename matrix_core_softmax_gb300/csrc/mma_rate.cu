// mma_rate.cu -- tensor-core rate probe: one CTA per SM issues block-scaled
// (or BF16) tcgen05 MMAs back to back from shared-memory operands into a TMEM
// accumulator, with nothing else to do, so that the measured rate is the
// ceiling the fused attention kernel's products are compared against.
//
// Kinds (fsa_probe_kind):
//   0  kind::mxf8f6f4, E4M3 x E4M3, M = 128, N = 256, K = 32 per instruction
//   1  kind::mxf8f6f4, E2M3 x E2M3, same shape (six-bit operands)
//   2  kind::mxf4,     E2M1 x E2M1 packed, M = 128, N = 256, K = 64, two E8M0
//      scales per row and instruction (scale_vec::2X)
//   3  the fused attention kernel's product pair per KV tile: the score
//      product (M = 128, N = 128, K = 128 in four E4M3 instructions, both
//      operands in shared memory) and the PV product (M = 128, N = D + 16 =
//      144, K = 128 in four instructions, A read from TMEM)
//   4  kind::f16, BF16 x BF16, M = 128, N = 256, K = 16 per instruction
// Operands hold pseudo-random finite values (the tensor core's power, and so
// the clock it sustains, depends on the data), scale bytes 2^-7 .. 2^7.
//
// Each CTA issues `iters` groups of four instructions (eight for kind 3) from
// one thread; every kRound groups it commits to one of two mbarriers and,
// before issuing further, waits (bounded) for the commit two rounds back, so
// at most two rounds are in flight.
#include "fsa_internal.h"
#include "sm100_ptx.cuh"

namespace fsa {
namespace {

constexpr int kProbeThreads = 128;
constexpr int kRound = 64;                  // instruction groups per commit
constexpr uint32_t kProbeCols = 512;
// TMEM columns: accumulator 0-255 (kind 3: S 0-127, O 256-399), P 400-431,
// scale atoms A 464, B 468 / 472 (rows 0-127 / 128-255), kind 3 P 476, V 480 / 484
constexpr uint32_t kPColP = 400, kPColSfA = 464, kPColSfB = 468, kPColSfP = 476, kPColSfV = 480;

struct __align__(1024) ProbeSmem {
    uint8_t a[128 * 128];  // 128 rows x 128 bytes, 128-byte swizzle atoms
    uint8_t b[256 * 128];  // 256 rows x 128 bytes
    uint8_t sf[4][kAtomBytes];
    uint64_t bar[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

__device__ __forceinline__ uint32_t mix32(uint32_t x) {
    x ^= x >> 16;
    x *= 0x7FEB352Du;
    x ^= x >> 15;
    x *= 0x846CA68Bu;
    x ^= x >> 16;
    return x;
}

// A byte of an operand of the given kind: any finite value of its type.
__device__ __forceinline__ uint8_t operand_byte(int kind, uint32_t i) {
    const uint32_t h = mix32(i * 0x9E3779B9u + 0x1234567u);
    if (kind == 4) {
        // bf16 halves: sign, exponent 120..134, any mantissa
        const uint32_t half = mix32(i >> 1);
        const uint32_t bits = (half & 0x807Fu) | ((120u + (half >> 8) % 15u) << 7);
        return static_cast<uint8_t>((i & 1) ? bits >> 8 : bits);
    }
    uint8_t b = static_cast<uint8_t>(h);
    if (kind == 0 || kind == 3) {
        if ((b & 0x7Fu) == 0x7Fu) b ^= 1u;  // no E4M3 NaN
    }
    return b;  // six- and four-bit types: every pattern is finite
}

__device__ __forceinline__ void mma_mxf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], [%6], p;\n\t"
        "}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
}

__global__ void __launch_bounds__(kProbeThreads, 1)
    mma_rate_kernel(int kind, int iters, uint64_t timeout_ns, unsigned int* err_word) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (smem_u32(smem_raw) & 1023u) {
        if (threadIdx.x == 0) atomicOr(err_word, kErrMisaligned);
        return;
    }
    ProbeSmem& sm = *reinterpret_cast<ProbeSmem*>(smem_raw);
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    if (warp == 0) {
        tmem_alloc(&sm.tmem_base, kProbeCols);
        tmem_relinquish();
    }
    for (uint32_t i = tid; i < sizeof(sm.a); i += kProbeThreads) sm.a[i] = operand_byte(kind, i);
    for (uint32_t i = tid; i < sizeof(sm.b); i += kProbeThreads)
        sm.b[i] = operand_byte(kind, i + 0x100000u);
    for (uint32_t i = tid; i < 4 * kAtomBytes; i += kProbeThreads)
        (&sm.sf[0][0])[i] = static_cast<uint8_t>(120u + mix32(i + 0x777u) % 15u);
    if (tid == 0) {
        sm.abort = 0;
        mbar_init(&sm.bar[0], 1);
        mbar_init(&sm.bar[1], 1);
        mbar_init(&sm.drain, 1);
        fence_mbar_init();
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    if (kind == 3) {
        // P of the PV product in TMEM: 128 rows x 128 E4M3 bytes (32 columns)
        uint32_t w[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            uint32_t x = mix32(static_cast<uint32_t>(tid * 32 + j) + 0xABCDu);
            x &= 0x77777777u;  // no E4M3 NaN in any byte
            w[j] = x;
        }
        tmem_st32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + kPColP, w);
        tmem_st_wait();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (tid == 0) {
        const uint64_t da = smem_desc(smem_u32(sm.a), 16, 1024, SWZ_128B);
        const uint64_t db = smem_desc(smem_u32(sm.b), 16, 1024, SWZ_128B);
        auto sfd = [&](int i) { return smem_desc(smem_u32(sm.sf[i]), 0, 128, SWZ_NONE); };
        // scale atoms into TMEM (A; B rows 0-127 and 128-255; P and V for kind 3)
        tc_cp_32x128b_x4(tmem + kPColSfA, sfd(0));
        tc_cp_32x128b_x4(tmem + kPColSfB, sfd(1));
        tc_cp_32x128b_x4(tmem + kPColSfB + 4, sfd(2));
        tc_cp_32x128b_x4(tmem + kPColSfP, sfd(3));
        tc_cp_32x128b_x4(tmem + kPColSfV, sfd(1));
        tc_cp_32x128b_x4(tmem + kPColSfV + 4, sfd(2));
        const uint32_t sfa = tmem + kPColSfA, sfb = tmem + kPColSfB;
#define FSA_SF(kk) ((static_cast<uint32_t>(kk) << 4) | (static_cast<uint32_t>(kk) << 29))
        const uint32_t id_e4m3 = idesc_mxf8f6f4(128, 256, 0, 0, 0, 0);
        const uint32_t id_e2m3 = idesc_mxf8f6f4(128, 256, 3, 3, 0, 0);
        // kind::mxf4: E2M1 (1) in the A and B format fields, UE8M0 scales
        const uint32_t id_mxf4 = (1u << 7) | (1u << 10) | (static_cast<uint32_t>(256 >> 3) << 17) |
                                 (1u << 23) | (static_cast<uint32_t>(128 >> 4) << 24);
        const uint32_t id_bf16 = idesc_bf16(128, 256, 0, 0);
        const uint32_t id_qk = idesc_mxf8f6f4(128, 128, 0, 0, 0, 0);
        const uint32_t id_pv = idesc_mxf8f6f4(128, 144, 0, 0, 0, 0);
        bool ok = true;
        for (int it = 0; ok && it < iters; ++it) {
            const int round = it / kRound;
            if (it % kRound == 0 && round >= 2 &&
                !mbar_wait(&sm.bar[round & 1], ((round - 2) >> 1) & 1, timeout_ns, &sm.abort)) {
                ok = false;
                break;
            }
            const uint32_t acc0 = it > 0 ? 1u : 0u;
            // four K steps of 32 bytes along the 128-byte rows
            switch (kind) {
                case 0:
                case 1: {
                    const uint32_t id = kind == 0 ? id_e4m3 : id_e2m3;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_mxf8f6f4(tmem, da + 2 * kk, db + 2 * kk, id | FSA_SF(kk), sfa, sfb,
                                     kk ? 1u : acc0);
                    break;
                }
                case 2:
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)  // scale bytes 0-1 or 2-3 of the atom
                        mma_mxf4(tmem, da + 2 * kk, db + 2 * kk,
                                 id_mxf4 | FSA_SF((kk & 1) * 2), sfa, sfb, kk ? 1u : acc0);
                    break;
                case 3:
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_mxf8f6f4(tmem, da + 2 * kk, db + 2 * kk, id_qk | FSA_SF(kk), sfa, sfb,
                                     kk ? 1u : acc0);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_mxf8f6f4_tmem_a(tmem + 256, tmem + kPColP + 8 * kk, db + 2 * kk,
                                            id_pv | FSA_SF(kk), tmem + kPColSfP, tmem + kPColSfV,
                                            kk ? 1u : acc0);
                    break;
                default:
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16(tmem, da + 2 * kk, db + 2 * kk, id_bf16, kk ? 1u : acc0);
                    break;
            }
            if ((it + 1) % kRound == 0) tc_commit(&sm.bar[round & 1]);
        }
#undef FSA_SF
        if (!ok) {
            sm.abort = 1;
            atomicOr(err_word, kErrTimeout);
        }
        // every product retired before TMEM is freed
        int dummy = 0;
        tc_commit(&sm.drain);
        if (!mbar_wait(&sm.drain, 0, timeout_ns, &dummy)) atomicOr(err_word, kErrTimeout);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kProbeCols);
    }
}

}  // namespace

// Floating-point operations of one launch: 2 M N K per instruction (kind 3:
// the attention metric's 4 * 128 * 128 * 128 per KV tile, the row-sum columns
// of the PV product not counted).
double mma_probe_flops(int kind, int ctas, int iters) {
    double per_group;
    switch (kind) {
        case 0:
        case 1: per_group = 4.0 * 2.0 * 128 * 256 * 32; break;
        case 2: per_group = 4.0 * 2.0 * 128 * 256 * 64; break;
        case 3: per_group = 4.0 * 128 * 128 * 128; break;
        default: per_group = 4.0 * 2.0 * 128 * 256 * 16; break;
    }
    return per_group * static_cast<double>(iters) * ctas;
}

cudaError_t launch_mma_probe(int kind, int ctas, int iters, uint64_t timeout_ns,
                             unsigned int* err_word, cudaStream_t st) {
    // more shared memory than two CTAs could share: one CTA per SM
    const int smem = 120 * 1024;
    static_assert(sizeof(ProbeSmem) <= 120 * 1024, "probe shared memory");
    cudaError_t e = cudaFuncSetAttribute(mma_rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    mma_rate_kernel<<<static_cast<unsigned>(ctas), kProbeThreads, smem, st>>>(kind, iters, timeout_ns,
                                                                              err_word);
    return cudaGetLastError();
}

}  // namespace fsa
