/*
 * attn.h -- C ABI of the GB300 (sm_103a) fused low-precision attention forward.
 *
 * The library computes the one-pass running-softmax attention forward over
 * 8-bit operands that its own quantiser produces:
 *
 *   attn_quantize  rotate (Q, K) and encode Q, K, V as E4M3 with per-block
 *                  scales or as MXFP8 with 32-element E8M0 scales
 *                  (attn_quantize_qkv: the three tensors in one launch)
 *   attn_fp8_fwd   S = Q K^T per key block, running row max and row sum,
 *                  P V accumulation, final normalisation and logsumexp;
 *                  FP32 softmax statistics, BF16 output
 *   attn_bf16_fwd  the same loop over BF16 operands (the accuracy comparator)
 *
 * Sources of the operations (page title, section):
 *   "Fused attention kernel" -- Overview (fused one-pass attention), 8-bit
 *     forward pass (e4m3, block quantisation, incoherent processing with a
 *     random sign diagonal times a Hadamard matrix), Implementation sketch
 *     (the running-softmax loop and its two notes).
 *   "FP8 attention that keeps FlashAttention-3 throughput at BF16-level
 *     accuracy" -- How it gets verified (E4M3 operands, FP32 softmax
 *     statistics, BF16 output, head dim 128, sequence 8192, causal and not).
 *   "FLAMIA: FLAsh MIcroscaling Attention for Fast and Causally Safe Training
 *     on Blackwell" -- Abstract and section 1 (token-block scaling, exact
 *     scaling options against causal leakage, document-local scaling of
 *     packed documents without repacking), section 2 (MX formats: 32-element
 *     blocks with a shared scale consumed by the block-scaled MMA), section
 *     4.3 (fused quantisation, longest-first ordering, folding score scales),
 *     appendix F (scales and work lists stay on the GPU, no host
 *     synchronisation, CUDA-graph capture, replay bitwise equal to eager).
 *
 * Conventions for every call:
 *   - Pointers are device pointers unless a comment says "host". The caller
 *     allocates and owns every buffer; the library never allocates or frees
 *     device memory and never synchronises the stream inside a call, so the
 *     calls can be captured in a CUDA graph.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy stream).
 *   - Argument errors are returned synchronously and nothing is launched.
 *     Errors found on the device (non-finite input, malformed cu_seqlens, a
 *     bounded wait that ran out) are OR-ed into a status word at the start of
 *     the caller's workspace and read back by attn_read_device_status.
 *   - Results are deterministic: the same inputs give bitwise the same
 *     outputs, eager or replayed from a graph.
 *   - Tensors Q, K, V, O are [total_tokens][heads][head_dim] with head_dim
 *     contiguous ("BSHD" packed; a batch of B sequences of N tokens is
 *     B documents of N tokens). Supported head_dim: 64 and 128 (MXFP8: 128).
 */
#ifndef PA_GB300_ATTN_H
#define PA_GB300_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The FP8 forward at head_dim 128 keeps, per query row, a reference maximum that
 * moves to the row's running maximum only when a key tile raises that by more
 * than this many log2 units (and always for the row's first key tile); the
 * probabilities 2^(s - m + 8) then stay below 2^8.75, inside E4M3's range, and
 * the output is rescaled only when the reference moves. 0 would be the exact
 * running maximum (the head_dim 64 and BF16 paths use that). */
#define ATTN_RESCALE_THRESHOLD 0.75f

/* How the FP8 forward at head_dim 128 forms each probability p = 2^x of the
 * softmax, x = s - m + 8 in log2 units (attn_fp8_fwd_ex; attn_fp8_fwd always
 * uses ATTN_EXP_HW). Source: FLAMIA section 1 (two bit-level exponentials for
 * inference), section 4.3 (log-domain probability quantisation) and section
 * 4.4 "Bit-Level Exponentials at Inference".
 *  ATTN_EXP_HW           the hardware exp2 (fp32, about 2 ulp), then E4M3 with
 *                        round to nearest even.
 *  ATTN_EXP_SCHRAUDOLPH  Schraudolph's exponential: the fp32 value whose bit
 *                        pattern is 2^23 (u + 127), u = x - ATTN_SCHRAUDOLPH_DELTA,
 *                        i.e. 2^floor(u) (1 + frac(u)), with u resolved to 2^-14
 *                        (round to nearest even) and limited to u >= -126; then
 *                        E4M3 with round to nearest even. The row sum adds the
 *                        fp32 values.
 *  ATTN_EXP_MITCHELL_P   log-domain P: the E4M3 code itself is the fixed-point
 *                        log2 of the probability (Mitchell: the code c of a
 *                        normal E4M3 value is 8 (log2 of its value + 7) where
 *                        the value is a power of two, linear in between), so
 *                        c = round(8 u + 56), limited to [0, 126]; the row sum
 *                        adds the exact E4M3 values of the codes.
 * Both bit-level modes shift x by ATTN_SCHRAUDOLPH_DELTA = log2(1/2 + 3 / (8 ln 2)),
 * the shift that minimises the root-mean-square relative error of the linear
 * interpolation between powers of two (1.77%, within -3.9% / +2.0%). */
typedef enum { ATTN_EXP_HW = 0, ATTN_EXP_SCHRAUDOLPH = 1, ATTN_EXP_MITCHELL_P = 2 } attn_exp_mode;
#define ATTN_SCHRAUDOLPH_DELTA 0.057984814725439975

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,     /* bad pointer, size, stride, alignment or combination */
    ATTN_ERR_UNSUPPORTED = 2,     /* valid request outside what the kernels implement */
    ATTN_ERR_CUDA = 3,            /* a CUDA runtime / driver call failed */
    ATTN_ERR_DEVICE_TIMEOUT = 4,  /* a bounded on-device wait ran out (kernel returned early) */
    ATTN_ERR_NONFINITE = 5,       /* a quantisation block held Inf or NaN */
    ATTN_ERR_SEED_MISMATCH = 6,   /* Q and K carry different rotations */
    ATTN_ERR_BAD_SEQLENS = 7,     /* cu_seqlens not 0 = c0 <= c1 <= ... = total_tokens */
    ATTN_ERR_WORKSPACE = 8        /* workspace NULL, misaligned or smaller than required */
} attn_status;

typedef enum { ATTN_IN_F32 = 0, ATTN_IN_BF16 = 1 } attn_in_dtype;

/* Scale layouts.
 * ATTN_E4M3_TOKBLOCK: E4M3 codes, one fp32 scale per (document, head, block of
 *   `block` consecutive tokens x head_dim); blocks start at the document start,
 *   the last one may be partial. scale = amax / 448, code = E4M3(x * (448 / amax)).
 *   block in {1, 32, 64, 128}; block 1 is the per-token scale of the
 *   causal-exact mode.
 *   Scales array: fp32 [heads][nb_cap], nb_cap = ceil(T / block) + num_docs;
 *   the block b of document i sits at column boff_i + b with
 *   boff_i = sum_{j < i} ceil(L_j / block).
 * ATTN_MX_ROW32 (Q, K): MXFP8, one E8M0 exponent per (token, head, 32
 *   consecutive channels); code = E4M3(x * 2^-X).
 * ATTN_MX_COL32 (V): MXFP8, one E8M0 exponent per (32 document-local tokens,
 *   head, channel): the 32-element blocks run along the sequence, the
 *   contraction axis of P V.
 *   MX scales array: bytes [heads][nt_cap][512], nt_cap = ceil(T/128) + num_docs,
 *   one 512-byte tile per (head, 128-token tile of a document), tile t of
 *   document i at index toff_i + t, toff_i = sum_{j < i} ceil(L_j / 128).
 *   Inside a tile, row r (ROW32: the token 128 t + r of the document; COL32:
 *   the channel r) and column group g (ROW32: channels 32 g..32 g + 31;
 *   COL32: tokens 128 t + 32 g..+31) hold the biased exponent X + 127 at byte
 *   (r % 32) * 16 + (r / 32) * 4 + g. Rows or groups past the document end
 *   hold 127. This is the order the block-scaled tensor-core MMA reads its
 *   scale factors in, so the forward copies tiles without reshuffling.
 * ATTN_MX_TOKEN (V of the causal-exact MX mode): MXFP8 codes with one E8M0
 *   exponent per (token, head) over all head_dim channels, so that no scale
 *   depends on another token; code = E4M3(x * 2^-X). Scales array: bytes
 *   [heads][T + num_docs], the token t (global index) at column t.
 * ATTN_NVFP4 (Q, K of the mixed NVFP4/FP8 path; head_dim 128, block 128):
 *   E2M1 codes, two per byte (the even channel in the low nibble), codes
 *   array [T][H][head_dim / 2]; an fp32 scale s_t = amax / (448 * 6) per
 *   (document, head, 128-token block) and an E4M3 scale per (token, head, 16
 *   consecutive channels): sf = E4M3(max |z|) with z = x * (448 / amax) over
 *   the 16 channels, code = E2M1(z * (6 / sf)) (0 where sf is 0); value =
 *   code * sf * s_t. Scales array: fp32 [heads][nt_cap] (block t of document
 *   i at toff_i + t, as the MX tiles), then, from byte offset
 *   ceil(heads * nt_cap * 4 / 1024) * 1024, bytes [heads][nt_cap][1024]: two
 *   512-byte tiles per 128-token block (channels 0..63, 64..127) in the MX
 *   tile order, row r (the token 128 t + r) and group g (16 channels) at
 *   byte (r % 32) * 16 + (r / 32) * 4 + g; rows past the document end hold 0.
 *   (FLAMIA sections 1 and 2: NVFP4 = 16-element blocks plus a tensor-level
 *   scale, here kept per document-local 128-token block.) */
typedef enum { ATTN_E4M3_TOKBLOCK = 0, ATTN_MX_ROW32 = 1, ATTN_MX_COL32 = 2, ATTN_MX_TOKEN = 3,
               ATTN_NVFP4 = 4 } attn_layout;

/* E8M0 exponent rule: NOSAT = smallest X with amax <= 448 * 2^X (nothing
 * saturates; default); OCP_FLOOR = floor(log2 amax) - 8 (values above
 * 448 * 2^X saturate). */
typedef enum { ATTN_MX_RULE_NOSAT = 0, ATTN_MX_RULE_OCP_FLOOR = 1 } attn_mx_rule;

typedef struct {
    int32_t total_tokens;          /* T >= 1 */
    int32_t heads;                 /* H >= 1 */
    int32_t head_dim;              /* d: 64 or 128 */
    int32_t num_docs;              /* >= 1; must be 1 when cu_seqlens is NULL */
    const int32_t* cu_seqlens;     /* device, num_docs + 1 prefix offsets, or NULL = one document */
} attn_shape;

/* A quantised operand. The caller sets codes, scales (buffers of the sizes
 * attn_quantize_sizes returns), layout, block and mx_rule before
 * attn_quantize; attn_quantize sets `rotated` and `hadamard_seed`. */
typedef struct {
    void* codes;                   /* device, [T][H][d] E4M3 bytes, 16-byte aligned */
    void* scales;                  /* device, see attn_layout; 16-byte aligned */
    int32_t layout;                /* attn_layout */
    int32_t block;                 /* tokens per scale block (ATTN_E4M3_TOKBLOCK) */
    int32_t mx_rule;               /* attn_mx_rule (MX layouts) */
    int32_t rotated;               /* 1 when codes are H_d * diag(signs) * x */
    uint64_t hadamard_seed;        /* seed of the sign diagonal when rotated */
} attn_qtensor;

/* Byte sizes of the code and scale buffers for one tensor of this shape.
 * Host-only; reads nothing on the device.
 * Source: "Fused attention kernel", 8-bit forward pass (one e4m3 code per
 * element, one scale per block); FLAMIA section 2 (one E8M0 scale per 32
 * elements). */
attn_status attn_quantize_sizes(const attn_shape* shape, int32_t layout, int32_t block,
                                size_t* codes_bytes, size_t* scales_bytes);

/* Workspace bytes that attn_quantize, attn_fp8_fwd and attn_bf16_fwd need for
 * this shape (one buffer serves all three; 256-byte aligned). Host-only.
 * Source: FLAMIA appendix F (work lists and scales kept on the GPU, so the
 * caller provides their memory once and no call allocates). */
attn_status attn_workspace_size(const attn_shape* shape, size_t* bytes);

/* The same size for a forward call of the given causality. The work list holds
 * one entry per (document, head, query-tile unit) whether or not the call is
 * causal, so `causal` does not change the result; it is accepted so that a
 * caller sizes the workspace for exactly the call it makes. Host-only.
 * Source: as attn_workspace_size. */
attn_status attn_fwd_workspace_size(const attn_shape* shape, int32_t causal, size_t* bytes);

/* Fused rotate-and-quantise, one kernel launch (each CTA builds the document
 * table it needs from cu_seqlens itself).
 * Source: "Fused attention kernel", 8-bit forward pass (e4m3 codes, block
 * quantisation, incoherent processing: a random sign diagonal times a
 * Hadamard matrix applied to Q and K, cancelling in Q K^T); FLAMIA section 2
 * (MX: 32-element blocks sharing one E8M0 scale), abstract and section 4.1
 * (document-local scales of packed documents, no repacking), section 4.3
 * (quantisation fused into one launch).
 * x: device, bf16 or fp32, element (t, h, c) at x[t * token_stride + h * head_stride + c]
 *    (strides in elements; channels contiguous; 16-byte aligned rows).
 * rotate != 0: codes of H_d * diag(s) * x, s_j = -1 if bit 63 of the j-th
 *    SplitMix64 output from `hadamard_seed` is set, else +1; H_d the
 *    unnormalised Sylvester Hadamard matrix, at d = 128 with its rows in the
 *    order the device transform leaves them: output channel p is Sylvester
 *    row pi(p), pi swapping the 3-bit fields at bits 1-3 and 4-6 of p (a
 *    Hadamard matrix still: H_d H_d^T = d I); at d = 64 the natural order.
 *    Q and K only; V is not rotated.
 * Writes out->codes and out->scales; sets out->rotated and out->hadamard_seed.
 * A scale block holding Inf or NaN raises ATTN_ERR_NONFINITE in the status word;
 * the codes and scale of such a block are then unspecified. */
attn_status attn_quantize(const void* x, int32_t in_dtype, int64_t token_stride, int64_t head_stride,
                          const attn_shape* shape, int32_t rotate, uint64_t hadamard_seed,
                          attn_qtensor* out, void* workspace, size_t workspace_bytes, void* stream);

/* Q, K and V in one launch: the same work as attn_quantize on each (Q and K
 * rotated with one seed when rotate != 0, V never), the three tensors' tiles
 * spread over one grid, so that the quantisation of a forward is a single
 * kernel (plus, above 64 documents, the document-table kernel once).
 * Source: FLAMIA section 4.3 (the quantisation of the forward's operands
 * fused into one launch); the operations as for attn_quantize.
 * q, k, v: device inputs of one dtype, one stride pair and the shape `shape`.
 * q_out, k_out, v_out: as attn_quantize's `out`; the layouts must be a set
 *    the forward takes: all ATTN_E4M3_TOKBLOCK with one block; ATTN_MX_ROW32
 *    for q and k with ATTN_MX_COL32 or ATTN_MX_TOKEN for v; ATTN_NVFP4 for q
 *    and k with ATTN_E4M3_TOKBLOCK block 128 for v. Any other set ->
 *    ATTN_ERR_INVALID_ARG; argument errors as attn_quantize, nothing launched.
 * Codes and scales are byte-identical to three attn_quantize calls with the
 * same arguments; device errors go to the one status word. */
attn_status attn_quantize_qkv(const void* q, const void* k, const void* v, int32_t in_dtype,
                              int64_t token_stride, int64_t head_stride, const attn_shape* shape,
                              int32_t rotate, uint64_t hadamard_seed, attn_qtensor* q_out,
                              attn_qtensor* k_out, attn_qtensor* v_out, void* workspace,
                              size_t workspace_bytes, void* stream);

/* FP8 attention forward over quantised operands.
 * Source: "Fused attention kernel", Implementation sketch (per key block:
 * S = Q K^T, new row max, rescale of the old sum and output by
 * exp(m_old - m_new), P V accumulation; one normalisation at the end and
 * lse = m + log l) and 8-bit forward pass (e4m3 operands, FP32 accumulation);
 * "FP8 attention that keeps FlashAttention-3 throughput at BF16-level
 * accuracy", How it gets verified (E4M3 operands, FP32 softmax statistics,
 * BF16 output, causal and non-causal); FLAMIA section 2 (block-scaled MMA),
 * section 4.3 (score scales folded into one multiplier, longest-first causal
 * work), sections 1 and 4.5 (exact scaling against causal leakage), section
 * 4.1 (packed documents).
 * q, k: ATTN_E4M3_TOKBLOCK, ATTN_MX_ROW32 or ATTN_NVFP4 (both the same; both
 *    rotated with the same seed or both not -> else ATTN_ERR_SEED_MISMATCH).
 * v: ATTN_E4M3_TOKBLOCK (with E4M3 q, k), or ATTN_MX_COL32 or ATTN_MX_TOKEN
 *    (with MX q, k), or ATTN_E4M3_TOKBLOCK with block 128 (with NVFP4 q, k:
 *    the mixed NVFP4/FP8 path of FLAMIA section 1, S from the block-scaled
 *    FP4 MMA, P V in E4M3; head_dim 128; causal_exact -> ATTN_ERR_UNSUPPORTED).
 * causal: key j > query i masked, positions local to each document.
 * causal_exact: requires causal, and block 1 for q, k and v (E4M3) or a v in
 *    ATTN_MX_TOKEN (MX: q and k rows are per token already); every scale then
 *    depends on its own token only, and V's scales are folded against a
 *    running maximum over positions <= i (for MX a power of two, exactly), so
 *    that no later token changes row i. An ATTN_MX_TOKEN v without
 *    causal_exact is folded against its document's largest scale.
 * softmax_scale <= 0 selects 1 / sqrt(d).
 * o: device bf16 [T][H][d]; lse: device fp32 [H][T], natural log of the
 *    scaled scores (lse_i = log sum_j exp(softmax_scale q_i . k_j)). */
attn_status attn_fp8_fwd(const attn_qtensor* q, const attn_qtensor* k, const attn_qtensor* v,
                         const attn_shape* shape, int32_t causal, int32_t causal_exact,
                         float softmax_scale, void* o, float* lse,
                         void* workspace, size_t workspace_bytes, void* stream);

/* attn_fp8_fwd with a choice of the probabilities' exponential (attn_exp_mode;
 * ATTN_EXP_HW is attn_fp8_fwd itself). The bit-level modes are inference
 * options: they need head_dim 128 and causal_exact = 0, and q, k, v either
 * all ATTN_E4M3_TOKBLOCK with block 128 or ATTN_MX_ROW32 q, k with an
 * ATTN_MX_COL32 v (else ATTN_ERR_UNSUPPORTED); an exp_mode outside the enum
 * is ATTN_ERR_INVALID_ARG. Every other argument, check and result is that of
 * attn_fp8_fwd; lse is the log of the row sum the mode forms.
 * Source: as attn_fp8_fwd, and FLAMIA sections 1, 4.3 and 4.4 (bit-level
 * exponentials at inference, log-domain probability quantisation). */
attn_status attn_fp8_fwd_ex(const attn_qtensor* q, const attn_qtensor* k, const attn_qtensor* v,
                            const attn_shape* shape, int32_t causal, int32_t causal_exact,
                            float softmax_scale, int32_t exp_mode, void* o, float* lse,
                            void* workspace, size_t workspace_bytes, void* stream);

/* BF16 attention forward: the same loop with bf16 q, k, v [T][H][d]
 * (contiguous), P in bf16, fp32 accumulation. Same o and lse as above.
 * Source: "FP8 attention that keeps FlashAttention-3 throughput at BF16-level
 * accuracy", The problem and How it gets verified (the BF16 attention whose
 * error the 8-bit path is measured against); "Fused attention kernel",
 * Implementation sketch (the loop). */
attn_status attn_bf16_fwd(const void* q, const void* k, const void* v, const attn_shape* shape,
                          int32_t causal, float softmax_scale, void* o, float* lse,
                          void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes that attn_bf16_bwd needs for this shape: the forward's
 * workspace plus two fp32 vectors per row (lse log2(e) and rowsum(dO o O)),
 * kept per (head, 128-token tile). 256-byte aligned; host-only.
 * Source: FLAMIA appendix F (scales and work lists on the GPU). */
attn_status attn_bwd_workspace_size(const attn_shape* shape, size_t* bytes);

/* BF16 attention backward: the gradients dq, dk, dv of o = softmax(scale q k^T) v
 * (causal mask and packed documents as in the forward) for an upstream
 * gradient dout. P is formed again from q, k and the forward's lse;
 * D = rowsum(dout o o) uses the forward's bf16 o. fp32 accumulation in the
 * tensor memory, P and dS rounded to bf16 as the operands of the dV, dK and dQ
 * products, bf16 outputs. Deterministic: every output element has one fixed
 * summation order, so repeated calls give the same bits.
 * q, k, v, o, dout: device bf16 [T][H][d], contiguous, 16-byte aligned;
 * lse: device fp32 [H][T] as attn_bf16_fwd writes it (natural log of the
 * scaled scores). dq, dk, dv: device bf16 [T][H][d], written for every token
 * of every document. head_dim 64 or 128.
 * softmax_scale <= 0 selects 1 / sqrt(d). Malformed cu_seqlens is reported
 * through the status word (ATTN_ERR_BAD_SEQLENS) and writes no gradient.
 * Source: FLAMIA section 1 (the forward and backward of the training call
 * over the same document-local token blocks), section 4.5 (the causal
 * backward); the gradients are the plain derivative of the forward's
 * definition ("Fused attention kernel", Overview). */
attn_status attn_bf16_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                          const float* lse, const attn_shape* shape, int32_t causal, float softmax_scale,
                          void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                          void* stream);

/* FP8 forward without a caller workspace (the pages have no counterpart to
 * this call). For callers that cannot allocate device memory where they run
 * attention -- a host that owns all device memory and forbids extra
 * allocations, a plugin inside another runtime's stream-ordered region, a
 * latency-critical path that must not risk an allocation that synchronises --
 * the scratch that attn_fp8_fwd keeps in its workspace lives here in one
 * file-scope device array of 16 MiB per device, held by every GPU that loads
 * the library until the process exits. Shapes whose attn_workspace_size
 * exceeds 16 MiB are refused with ATTN_ERR_UNSUPPORTED; nothing is allocated.
 * The first call on a device (with that device current) looks up the array's
 * address; make it before any stream capture. All calls share the array:
 * calls that overlap on the GPU race. Arguments and results are those of
 * attn_fp8_fwd, and so are its argument checks, made before the array or
 * `status` is touched. `status` (device, may be NULL) receives the forward's
 * device status word (bit e = attn_status e), cleared at the start of the
 * call; it is written only when the call returns ATTN_OK. Errors that the
 * quantiser found (a non-finite block) stay in the workspace given to
 * attn_quantize, not here. */
attn_status attn_fp8_fwd_noalloc(const attn_qtensor* q, const attn_qtensor* k, const attn_qtensor* v,
                                 const attn_shape* shape, int32_t causal, int32_t causal_exact,
                                 float softmax_scale, void* o, float* lse, uint32_t* status, void* stream);

/* Synchronises `stream`, reads and clears the device status word in
 * `workspace`, and returns the first error it holds (ATTN_OK if none).
 * flags_out (host, may be NULL) receives the raw bit set (bit e = error e).
 * Source: FLAMIA appendix F (no host synchronisation inside the calls: the
 * errors found on the device wait in the workspace until the caller asks). */
attn_status attn_read_device_status(void* workspace, void* stream, uint32_t* flags_out);

/* Limit, in SM clock cycles, of every bounded on-device wait of the attention
 * calls made after this one (default about 2 s of SM clock; cycles <= 0
 * restores it). When a wait runs out the kernel stops its work, lets the copies
 * and MMAs already in flight finish, frees what it holds and returns; the call's
 * status word then holds ATTN_ERR_DEVICE_TIMEOUT and O and lse are undefined.
 * A short limit makes that path testable without a device fault. Process-wide;
 * host only (never touches the device). Returns ATTN_OK. No counterpart on the
 * pages: the bounded waits are this library's failure detection. */
attn_status attn_set_wait_limit(int64_t cycles);

/* Work order of the FP8 forward's pair kernel (head_dim 128) for the calls
 * made after this one. ATTN_SCHED_STATIC (default): each CTA takes rounds of
 * the longest-first work list, in alternating directions for causal work.
 * ATTN_SCHED_TICKET: each CTA takes its next item just in time from a global
 * counter in the workspace, the items in list order (longest first for causal
 * work). The results are bitwise the same; only which CTA computes which item
 * changes. Process-wide; host only. Returns ATTN_ERR_INVALID_ARG for any
 * other value. Source: FLAMIA section 4.3 (just-in-time work acquisition by
 * cluster launch control, against a static longest-first order). */
typedef enum { ATTN_SCHED_STATIC = 0, ATTN_SCHED_TICKET = 1 } attn_schedule;
attn_status attn_set_schedule(int32_t schedule);

/* Static description of a status code (no counterpart on the pages). */
const char* attn_status_string(int32_t status);

/* Number of streaming multiprocessors the forward sizes its persistent grid
 * for on the current device, or -1 on error (no counterpart on the pages). */
int32_t attn_device_sm_count(void);

#ifdef __cplusplus
}
#endif
#endif
