/*
 * fsa.h -- C ABI of the GB300 (sm_103a) Fused-Softmax quantized attention
 * library, libfsa.so.
 *
 * What the library computes is the forward pass described in
 *   "Fused-Softmax shifts an AI attention bottleneck onto faster GPU
 *    hardware" (article on arXiv:2611.09225), paragraphs 5-8, and
 *   "Fused softmax makes quantized attention faster on AMD GPUs", section
 *    "What the evidence shows", bullet "Move work, keep correction":
 *   Q, K, V are microscaled (32-element blocks sharing one E8M0 power-of-two
 *   scale) to MXFP8, MXFP6 or MXFP4; S = Q K^T runs on block-scaled tensor
 *   cores with the frozen row-max subtraction and the Schraudolph
 *   exponential's affine map applied to the accumulator; the rounded result
 *   is reinterpreted as a BF16 weight, converted a second time into an MX
 *   operand P, and O = P V and l = P 1 both come from tensor-core products on
 *   that same P.  A gate rolls the reference maximum forward when a tile's
 *   scores pass it by more than a threshold and rescales O and l.
 *
 * Conventions shared by every call:
 *  - All tensor pointers are DEVICE pointers owned by the caller, 16-byte
 *    aligned.  Attention tensors are bf16, contiguous [B][H][S][D] ("BHSD").
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Work is enqueued asynchronously on it; a call returns after
 *    launching.  Argument errors are detected on the host and returned before
 *    anything is launched.
 *  - Device-side failures that the kernels detect themselves (a bounded wait
 *    that ran out) are recorded in a per-device error word; read and clear it
 *    with fsa_get_device_error().
 *  - Only sm_103a (GB300) and sm_100a devices are supported; others get
 *    FSA_ERR_UNSUPPORTED.
 *  - Inputs must be finite; the output is undefined for Inf or NaN inputs.
 */
#ifndef FSA_H_
#define FSA_H_

#include <stdint.h>

#if defined(__GNUC__)
#define FSA_API __attribute__((visibility("default")))
#else
#define FSA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Attention formats ("Fused-Softmax shifts ...", paragraph 8): element type
 * of Q/K/V and of P.  MXFP8: E4M3 / E4M3.  MXFP6: E2M3 / E2M3.
 * MXFP4: E2M1 / E2M3 (the MXFP4 variant keeps six-bit P). */
typedef enum {
    FSA_MXFP8 = 0,     /* E4M3 Q/K/V, E4M3 P */
    FSA_MXFP6 = 1,     /* E2M3 Q/K/V, E2M3 P */
    FSA_MXFP4 = 2,     /* E2M1 Q/K/V, six-bit E2M3 P */
    /* E2M1 Q/K/V with the EFQ-Softmax P producer ("EFQ-Softmax: Exp-Free
     * Quantization for Softmax", sections B-C and "A. Integration with Online
     * Attention"): online attention with the running row maximum (O and l
     * rescaled exactly when it grows; no rollback gate, `threshold` is
     * ignored and no firings are reported) and E2M1 P generated directly
     * from the shifted scores: per 32-key block, u = (s - m) log2(e), scale
     * 2^X with X = ceil(max u - log2 6), code = clip(floor((u - X - tau) /
     * h), 0, 7); the same P feeds O and l.  tau, h: fsa_options. */
    FSA_MXFP4_EFQ = 3
} fsa_format;

/* Element types of fsa_quantize_mx. */
typedef enum { FSA_ELEM_E4M3 = 0, FSA_ELEM_E2M3 = 1, FSA_ELEM_E2M1 = 2 } fsa_elem;

typedef enum {
    FSA_OK = 0,
    FSA_ERR_INVALID_ARGUMENT = 1, /* null pointer, bad size, bad enum, theta */
    FSA_ERR_UNSUPPORTED = 2,      /* device architecture or head dim D */
    FSA_ERR_CUDA = 3,             /* a CUDA runtime/driver call failed */
    FSA_ERR_OUT_OF_MEMORY = 4,    /* workspace allocation failed */
    FSA_ERR_TIMEOUT = 5           /* a kernel's bounded wait ran out */
} fsa_status;

/* Debug switches of fsa_options.debug_flags (test use only). */
#define FSA_DEBUG_SKIP_KV_ARRIVE 0x1 /* the loader never signals KV tile 1:
                                        the consumers' bounded waits run out,
                                        the kernel exits cleanly and the error
                                        word reads FSA_ERR_TIMEOUT */

typedef struct {
    /* Score scale; <= 0 selects 1/sqrt(D). */
    float sm_scale;
    /* Optional device output, [B*H*S][n_t] bytes with n_t = ceil(S/128):
     * byte (row, t) is set to 1 when the rollback gate fired for that row at
     * KV tile t (tile 0 initialises the reference and never fires) and to 0
     * otherwise.  NULL: not written. */
    uint8_t *rollback_bits;
    /* Optional device counter; the number of gate firings is ADDED to it.
     * NULL: not written. */
    unsigned long long *rollback_count;
    /* Optional caller-owned device workspace of at least
     * fsa_attention_workspace_size() bytes, 256-byte aligned.  NULL: the
     * library uses its own cached per-device workspace (allocated on first
     * use and grown as needed; concurrent calls on different streams must
     * then not overlap). */
    void *workspace;
    uint64_t workspace_bytes;
    /* Bounded-wait limit of the kernels in milliseconds; <= 0 means 2000. */
    int wait_timeout_ms;
    int debug_flags;
    /* FSA_MXFP4_EFQ's affine rule; efq_h <= 0 selects the library's offline
     * calibration, tau = -2.44, h = 0.61 (the pages print no values). */
    float efq_tau;
    float efq_h;
    /* Host-buffer entry points only: nonzero declares q, k, v final when the
     * call is made (nothing enqueued earlier on `stream` writes them), so
     * their copy-in may start at once instead of after the work already on
     * `stream` -- consecutive calls then overlap their copies.  0: the
     * copies wait for that work. */
    int host_inputs_ready;
    /* Rollback gate ("Fused-Softmax shifts ...", paragraph 12): 0, the
     * method's gate on the FP32 scores (a tile whose row maximum passes the
     * reference by more than `threshold` rolls back); 1, the shortcut the
     * pages' fastest four-bit kernel takes, gating on converted values: a tile
     * rolls back when its largest P block scale under the current reference
     * exceeds the scale of threshold's own weight code.  The shortcut is the
     * FP32 gate at a threshold raised to the end of that scale's binade, so
     * it misses the firings whose excess lies between the two.  Ignored by
     * FSA_MXFP4_EFQ; other values: FSA_ERR_INVALID_ARGUMENT. */
    int gate_mode;
} fsa_options;

/*
 * fsa_quantize_mx -- MX microscaling of a bf16 tensor x[batch][rows][cols].
 *
 * Source: "EFQ-Softmax: Exp-Free Quantization for Softmax", section
 * "B. Block-Scaled E2M1 Probability Representation" (blocks sharing an
 * exponent-only E8M0 scale) and "Fused-Softmax shifts ...", paragraphs 7-8
 * (MXFP8/MXFP6/MXFP4 operands).  Scale rule (the pages print none; this is
 * the library's reading): for a block with largest magnitude amax the scale
 * is 2^X with X the smallest integer such that amax <= max_elem * 2^X,
 * clamped to [-127, 127]; an all-zero block has X = -127.  Elements are
 * x / 2^X rounded to nearest, ties to even (never saturating by
 * construction).
 *
 *  block_axis = 1: blocks of 32 run along cols (Q and K: along D).
 *      codes [batch][rows][cols], scales [batch][rows][ceil(cols/32)].
 *  block_axis = 0: blocks of 32 run along rows and the output is transposed
 *      (V: along the keys).  codes [batch][cols][rows],
 *      scales [batch][cols][ceil(rows/32)].
 *  The last block of a line may be shorter than 32.
 *  codes: one element code per byte in the low bits (E4M3: 8 bits, E2M3:
 *         6 bits, E2M1: 4 bits), sign in the code's top bit.
 *  scales: E8M0 bytes, X + 127.
 *  All three pointers are device pointers; x must be 16-byte aligned when
 *  block_axis = 1 and cols % 8 == 0 (otherwise 2-byte aligned suffices).
 * Returns FSA_ERR_INVALID_ARGUMENT for null pointers, negative sizes, a bad
 * elem_fmt or block_axis; FSA_OK for an empty tensor (nothing launched).
 */
FSA_API fsa_status fsa_quantize_mx(const void *x, int64_t batch, int64_t rows, int64_t cols,
                           int block_axis, int elem_fmt, uint8_t *codes, uint8_t *scales,
                           void *stream);

/*
 * fsa_attention_fwd -- Fused-Softmax MX attention forward, non-causal,
 * Sq = Sk = S.  q, k, v, o: bf16 device tensors [B][H][S][D].
 *
 * Per query row i and KV tile t of 128 keys ("Fused-Softmax shifts ...",
 * paragraphs 5 and 6):
 *   s_ij = sm * q^_i . k^_j (block-scaled MMA, FP32 accumulate);
 *   tile 0 freezes m_i = max_j s_ij;  a later tile whose max passes m_i by
 *   more than `threshold` rolls back: O_i, l_i *= exp(m_i - m'), m_i = m';
 *   y_ij = 128 * ((s_ij - m_i) * log2(e) + 127) - 7;  code = clamp(rne(y), 0,
 *   0x7F7F) read as a bf16 p_ij;  P^ = MX(p) in 32-key blocks (E4M3 for
 *   MXFP8, E2M3 otherwise);  O_i += P^ V^, l_i += P^ 1 (both MMAs);
 *   o_i = bf16(O_i / l_i).  Keys >= S are masked before the gate.
 * Requirements: B, H, S >= 1; D in {64, 128}; threshold finite in [0, 80]
 * (128 * (threshold * log2(e) + 127) must stay a finite bf16 code).
 * Uses the library's cached workspace (see fsa_options.workspace).
 */
FSA_API fsa_status fsa_attention_fwd(const void *q, const void *k, const void *v, void *o,
                             int B, int H, int S, int D, int fmt, float threshold,
                             void *stream);

/* As fsa_attention_fwd with options (NULL = defaults). */
FSA_API fsa_status fsa_attention_fwd_ex(const void *q, const void *k, const void *v, void *o,
                                int B, int H, int S, int D, int fmt, float threshold,
                                const fsa_options *opt, void *stream);

/*
 * fsa_cross_attention_fwd -- fsa_attention_fwd_ex with queries and keys of
 * different lengths (cross-attention shapes): q and o are bf16 device
 * tensors [B][H][Sq][D], k and v [B][H][Sk][D].  Every query row runs the
 * same per-row method over the Sk keys in KV tiles of 128 (tile 0 of the keys
 * freezes the reference, keys >= Sk are masked); rows are independent, so
 * with Sq = Sk this is exactly fsa_attention_fwd_ex.  The pages measure
 * self-attention only ("Fused-Softmax shifts ...", paragraph 9: only
 * self-attention was swapped in the video model); this entry point is the
 * library's generalisation.  opt->rollback_bits, when given, is
 * [B*H*Sq][ceil(Sk/128)]; opt->workspace, when given, needs
 * fsa_cross_attention_workspace_size() bytes.  Requirements as for
 * fsa_attention_fwd with Sq, Sk >= 1.
 */
FSA_API fsa_status fsa_cross_attention_fwd(const void *q, const void *k, const void *v, void *o,
                                           int B, int H, int Sq, int Sk, int D, int fmt,
                                           float threshold, const fsa_options *opt, void *stream);

/* Bytes of device workspace fsa_cross_attention_fwd needs (MX copies of Q,
 * K, V and their scales).  0 for invalid arguments. */
FSA_API uint64_t fsa_cross_attention_workspace_size(int B, int H, int Sq, int Sk, int D, int fmt);

/* The two halves of fsa_cross_attention_fwd, as fsa_attention_prepare /
 * fsa_attention_run below with q [B][H][Sq][D] and k, v [B][H][Sk][D]; the
 * workspace needs fsa_cross_attention_workspace_size() bytes. */
FSA_API fsa_status fsa_cross_attention_prepare(const void *q, const void *k, const void *v, int B,
                                               int H, int Sq, int Sk, int D, int fmt,
                                               void *workspace, uint64_t workspace_bytes,
                                               void *stream);
FSA_API fsa_status fsa_cross_attention_run(const void *workspace, uint64_t workspace_bytes, void *o,
                                           int B, int H, int Sq, int Sk, int D, int fmt,
                                           float threshold, const fsa_options *opt, void *stream);

/*
 * The two halves of fsa_attention_fwd_ex, for callers that keep the MX
 * copies (e.g. quantize K/V once and attend many times) or time the parts.
 *
 * fsa_attention_prepare: MX-quantizes q, k, v (bf16 [B][H][S][D]) into the
 * caller's device workspace (>= fsa_attention_workspace_size() bytes,
 * 256-byte aligned): Q and K in 32-element blocks along D, V in 32-key
 * blocks along the keys, stored transposed; element type per `fmt`.
 * fsa_attention_run: the fused attention kernel on a prepared workspace;
 * shape and fmt must be those given to fsa_attention_prepare; opt may be
 * NULL; opt->workspace is ignored.
 */
FSA_API fsa_status fsa_attention_prepare(const void *q, const void *k, const void *v, int B, int H,
                                         int S, int D, int fmt, void *workspace,
                                         uint64_t workspace_bytes, void *stream);
FSA_API fsa_status fsa_attention_run(const void *workspace, uint64_t workspace_bytes, void *o,
                                     int B, int H, int S, int D, int fmt, float threshold,
                                     const fsa_options *opt, void *stream);

/* Bytes of device workspace fsa_attention_fwd needs for this shape (MX
 * copies of Q, K, V and their scales, and for MXFP6 / MXFP4 the row-norm
 * bounds of the quantized Q and K).  0 for invalid arguments. */
FSA_API uint64_t fsa_attention_workspace_size(int B, int H, int S, int D, int fmt);

/*
 * fsa_bf16_attention_fwd -- conventional BF16 flash attention (exact
 * softmax with a running maximum, FP32 accumulation, BF16 P), the speed
 * and error denominator the pages compare against ("Fused-Softmax shifts
 * ...", paragraphs 7-8).  Same tensor conventions; D in {64, 128}.
 */
FSA_API fsa_status fsa_bf16_attention_fwd(const void *q, const void *k, const void *v, void *o,
                                  int B, int H, int S, int D, void *stream);

/*
 * fsa_attention_fwd_noalloc -- fsa_attention_fwd without any device memory
 * allocation.  (An addition of this library; the pages have no counterpart.)
 *
 * For callers that must not allocate or free device memory once they are
 * running -- for example code whose device memory budget is owned entirely by
 * its own allocator, or a latency-critical loop that cannot afford
 * cudaMalloc/cudaFree (which may synchronise the device or fail under memory
 * pressure).  Instead of the cached workspace, the MX copies of q, k, v live in
 * a fixed 64 MiB array compiled into the library: every device that loads the
 * library holds it until the process exits.
 *  - Same arguments, layouts and results as fsa_attention_fwd.
 *  - Shapes whose workspace (fsa_attention_workspace_size) exceeds 64 MiB --
 *    roughly B*H*S*D above 21 million -- return FSA_ERR_INVALID_ARGUMENT.
 *  - The first call on a device looks up the array's device address (and
 *    that of a status word beside it) with that device current; make that
 *    first call before any stream capture.
 *  - All calls on a device share the one array, which keeps the last call's
 *    contents: calls that overlap on the GPU (different streams, or several
 *    host threads) race on it and must be serialised by the caller.
 *  - A kernel whose bounded wait ran out sets the status word beside the
 *    array (a static device object, zero at load); fsa_get_device_error
 *    reads and clears it together with the other entry points' word and
 *    allocates nothing, so these callers can use it too.
 */
FSA_API fsa_status fsa_attention_fwd_noalloc(const void *q, const void *k, const void *v, void *o,
                                             int B, int H, int S, int D, int fmt,
                                             float threshold, void *stream);

/*
 * fsa_attention_fwd_host / fsa_cross_attention_fwd_host -- the fused
 * attention on HOST buffers.  (An addition of this library; the pages have
 * no counterpart.)
 *
 * q, o: host bf16 [B][H][Sq][D]; k, v: host bf16 [B][H][Sk][D] (Sq = Sk = S
 * for the self-attention form).  Same formats, threshold, options and
 * results as fsa_cross_attention_fwd; opt->rollback_bits and
 * opt->rollback_count stay DEVICE pointers, opt->workspace is ignored.
 *  - The heads are streamed through the device in chunks (about eight, each
 *    at least two waves of query tiles): while one chunk's quantizer and
 *    fused kernel run, the next chunk's q, k, v are copied in and the
 *    previous chunk's output copied out, on two copy streams of the library;
 *    consecutive chunks compute on `stream` and on a second stream of the
 *    library, so that their kernels overlap.
 *  - Page-locked host memory (cudaHostAlloc, cudaHostRegister) lets the
 *    copies run asynchronously and overlap; pageable memory gives the same
 *    results with copies that block the calling thread.
 *  - Asynchronous like the other calls: the work is ordered after what was
 *    already enqueued on `stream`, and `stream` waits for all of it, so o is
 *    complete once `stream` has been synchronised.  The caller keeps q, k,
 *    v unchanged and o unread until then.
 *  - Device memory: two chunk buffer sets (bf16 inputs and output of a
 *    chunk plus its MX workspace), cached per device, grown on demand
 *    (synchronising), freed by fsa_release_workspace.  Host-side use is
 *    serialised by a per-device lock; calls on different streams are
 *    ordered on the GPU through the library's events.
 *  - Errors: as fsa_cross_attention_fwd (no pointer alignment is required
 *    of the host buffers); FSA_ERR_OUT_OF_MEMORY if the chunk buffers cannot
 *    be allocated, FSA_ERR_CUDA if a copy, event or launch fails.
 */
FSA_API fsa_status fsa_attention_fwd_host(const void *q, const void *k, const void *v, void *o,
                                          int B, int H, int S, int D, int fmt, float threshold,
                                          const fsa_options *opt, void *stream);
FSA_API fsa_status fsa_cross_attention_fwd_host(const void *q, const void *k, const void *v, void *o,
                                                int B, int H, int Sq, int Sk, int D, int fmt,
                                                float threshold, const fsa_options *opt,
                                                void *stream);

/*
 * fsa_mma_rate_probe -- the tensor-core rate the fused kernel is measured
 * against.  (A measurement aid of this library, not part of the method; the
 * pages compare their kernels' speed only with BF16 attention, "Fused-Softmax
 * shifts ...", paragraph 8, and print no peak.)
 *
 * Launches `ctas` CTAs (one per SM: pass the SM count) that each issue
 * `iters` groups of tensor-core products back to back, with operands of
 * pseudo-random finite values already in shared memory and tensor memory and
 * nothing else to do, on `stream`; the caller times the launch.
 *  kind 0: kind::mxf8f6f4 block-scaled MMA, E4M3 x E4M3, M = 128, N = 256,
 *          four K = 32 instructions per group;
 *  kind 1: the same with E2M3 x E2M3 (six-bit) operands;
 *  kind 2: kind::mxf4, packed E2M1 x E2M1, M = 128, N = 256, four K = 64
 *          instructions per group (two E8M0 scales per row and instruction);
 *  kind 3: the fused attention kernel's products of one KV tile: the score
 *          product (M = N = 128, K = 128, E4M3, operands in shared memory)
 *          and the PV product (M = 128, N = 144 = D + 16, K = 128, A from
 *          tensor memory);
 *  kind 4: kind::f16 BF16 x BF16, M = 128, N = 256, four K = 16 instructions.
 * *flops_per_launch (host, may be NULL) receives the launch's floating-point
 * operations: 2 M N K per instruction; kind 3 the attention metric's
 * 4 * 128 * 128 * 128 per group (the 16 row-sum columns not counted).
 * Returns FSA_ERR_INVALID_ARGUMENT for kind outside 0..4, ctas outside
 * 1..65535 or iters outside 1..2^24.  A bounded wait that ran out is reported
 * by fsa_get_device_error.
 */
FSA_API fsa_status fsa_mma_rate_probe(int kind, int ctas, int iters, double *flops_per_launch,
                                      void *stream);

/* Synchronises `stream`, then reads and clears the device error words of the
 * current device (the allocating entry points' word and, once that entry
 * point has run there, fsa_attention_fwd_noalloc's): FSA_OK, FSA_ERR_TIMEOUT,
 * or FSA_ERR_CUDA if the sync itself failed.  Allocates no device memory. */
FSA_API fsa_status fsa_get_device_error(void *stream);

/* Static description of a status code. */
FSA_API const char *fsa_status_string(fsa_status s);

/* Frees the library's cached workspaces (including the host-buffer entry
 * points' chunk buffers) on every device (synchronising). */
FSA_API void fsa_release_workspace(void);

#ifdef __cplusplus
}
#endif
#endif /* FSA_H_ */
