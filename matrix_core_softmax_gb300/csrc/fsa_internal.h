// fsa_internal.h -- declarations shared by the library's translation units.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fsa {

// Element formats (match fsa_elem).
enum Elem : int { ELEM_E4M3 = 0, ELEM_E2M3 = 1, ELEM_E2M1 = 2 };

// Output layout of the quantizer.
//  PLAIN: element codes of the format, plain row-major scale bytes.
//  ATTN:  E4M3 bit patterns of the quantized elements (every E2M3 / E2M1
//         value is exactly an E4M3 value) and scale bytes packed into the
//         128-row x 4-block "scale atoms" the tensor core's scale-factor
//         copy expects: for row r of a 128-row tile and block kb (< 4),
//         byte (r % 32) * 16 + (r / 32) * 4 + kb of the tile's 512 bytes.
enum QuantLayout : int { QL_PLAIN = 0, QL_ATTN = 1 };

constexpr int kTile = 128;        // query rows / keys per tile
constexpr int kAtomBytes = 512;   // scale atom of one 128-row tile

// Workspace of the fused attention call: MX copies of Q, K, V and scales
// (Sq query rows and Sk keys per head; Sq = Sk for self-attention).
struct AttnWorkspace {
    uint8_t* qc;   // [BH][Sq][D]  E4M3 bit patterns
    uint8_t* kc;   // [BH][Sk][D]
    uint8_t* vt;   // [BH][D][Sk16] V transposed, keys contiguous, Sk16 = round_up(Sk, 16)
    uint8_t* qsf;  // [BH][ceil(Sq/128)][512] atoms, rows = query rows
    uint8_t* ksf;  // [BH][ceil(Sk/128)][512] atoms, rows = keys
    uint8_t* vsf;  // [BH][ceil(Sk/128)][512] atoms, rows = d, blocks along keys
    size_t sf_bytes_total;  // qsf..vsf are contiguous
    float* qnorm;  // [BH][Sq] upper bound of |q^_i| (six-bit formats)
    float* knorm;  // [BH][ceil(Sk/128)] per KV tile: max over its keys of an upper bound of |k^_j|
};
size_t attn_workspace_bytes(int64_t BH, int64_t Sq, int64_t Sk, int D);
AttnWorkspace attn_workspace_carve(void* base, int64_t BH, int64_t Sq, int64_t Sk, int D);

// Row-norm output of the row quantizer (ATTN layout only): none, an upper
// bound of the Euclidean norm of every quantized row, or per 128-row tile the
// largest of those bounds (atomic maximum into a zeroed array).
enum NormMode : int { NORM_NONE = 0, NORM_ROW = 1, NORM_TILE_MAX = 2 };

// Quantizer launchers (quantize.cu).
cudaError_t launch_quant_rows(const uint16_t* x, int64_t lines, int64_t cols, int elem,
                              int layout, uint8_t* codes, uint8_t* scales, int64_t rows_per_mat,
                              cudaStream_t st, float* norms = nullptr, int norm_mode = NORM_NONE);
cudaError_t launch_quant_cols(const uint16_t* x, int64_t batch, int64_t rows, int64_t cols,
                              int elem, int layout, uint8_t* codes, int64_t code_pitch,
                              uint8_t* scales, cudaStream_t st);

// Attention launchers.
struct AttnLaunch {
    const CUtensorMap* tm_q;
    const CUtensorMap* tm_k;
    const CUtensorMap* tm_v;
    AttnWorkspace ws;
    void* o;
    int64_t BH;
    int Sq, Sk, D, fmt;  // query rows and keys per head
    float sm_scale, threshold;
    float efq_tau, efq_h;  // EFQ affine rule (fmt 3)
    uint8_t* rollback_bits;
    unsigned long long* rollback_count;
    uint64_t timeout_ns;
    int debug_flags;
    int gate_mode;  // 0: FP32 gate, 1: shortcut on the P block scale
    unsigned int* err_word;
};
cudaError_t launch_fsa_attention(const AttnLaunch& a, cudaStream_t st);

struct Bf16Launch {
    const CUtensorMap* tm_q;
    const CUtensorMap* tm_k;
    const CUtensorMap* tm_v;
    void* o;
    int64_t BH;
    int S, D;
    float sm_scale;
    uint64_t timeout_ns;
    unsigned int* err_word;
};
cudaError_t launch_bf16_attention(const Bf16Launch& a, cudaStream_t st);

// Tensor-core rate probe (mma_rate.cu).
double mma_probe_flops(int kind, int ctas, int iters);
cudaError_t launch_mma_probe(int kind, int ctas, int iters, uint64_t timeout_ns,
                             unsigned int* err_word, cudaStream_t st);

// Device error word codes.
constexpr unsigned int kErrTimeout = 1u;
constexpr unsigned int kErrMisaligned = 2u;  // shared-memory base not 1024-byte aligned

}  // namespace fsa
