/*
 * attn_oracle.h -- CPU oracle for the fused low-precision attention forward pass.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline / reference leg may load or call this code. The
 * product library (the CUDA path) never includes, links or loads it, and the
 * two share no code, header, table or constant generator.
 *
 * Three parts, each written from the pages it cites:
 *   O-1  FP64 softmax attention, the plain definition
 *        ("Fused attention kernel", Overview; the FP64 reference of the
 *        "8-bit forward pass (FP8, Hopper)" section; "FP8 attention that keeps
 *        FlashAttention-3 throughput at BF16-level accuracy", How it gets
 *        verified).
 *   O-2  Bit-level quantiser: random-sign diagonal x Hadamard rotation of Q
 *        and K, block scales (E4M3 token blocks) or 32-element E8M0 scales
 *        (MXFP8), E4M3 encoding ("Fused attention kernel", 8-bit forward pass:
 *        block quantisation, incoherent processing; FLAMIA, section 2
 *        Background: microscaling).
 *   O-3  Quantised-operand emulation of the running-softmax loop, key blocks
 *        of 128 in ascending order ("Fused attention kernel", Implementation
 *        sketch, with both of its notes applied).
 *
 * Pins: every function here is checked by tests marked "not gpu" against
 * something other than itself (brute force, closed forms, textbook identities,
 * a published generator test vector). The one part left without a pin is the
 * pages' printed RMSE pair (2.4e-2 / 9.1e-3): parity unpinned, used as a trend
 * check only, because the pages do not give its generator.
 */
#ifndef ATTN_ORACLE_H
#define ATTN_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { OR_E4M3_TOKBLOCK = 0, OR_MX_ROW32 = 1, OR_MX_COL32 = 2, OR_MX_TOKEN = 3, OR_NVFP4 = 4 };
enum { OR_MX_RULE_NOSAT = 0, OR_MX_RULE_OCP_FLOOR = 1 };
enum { OR_OK = 0, OR_ERR_ARG = 1, OR_ERR_NONFINITE = 5 };

/* threads used by the parallel loops (0 = all online host cores) */
int or_set_threads(int n);
int or_threads(void);

/* ---- number formats ---- */
double   or_e4m3_decode(uint8_t code);
uint8_t  or_e4m3_encode(float x);
double   or_e2m1_decode(uint8_t code);   /* low 4 bits: sign, 2 exponent bits (bias 1), 1 mantissa bit */
uint8_t  or_e2m1_encode(float x);        /* nearest of 0, 0.5, 1, 1.5, 2, 3, 4, 6, ties to even, beyond 6 -> 6 */
int      or_e8m0_exponent(float amax, int rule);   /* unbiased X; byte = X + 127 */
uint16_t or_bf16_rne(float x);
void     or_e4m3_encode_range(uint64_t start, uint64_t count, uint8_t* out); /* bit patterns start.. */

/* ---- rotation ---- */
uint64_t or_splitmix64_next(uint64_t* state);
void     or_signs(uint64_t seed, int d, float* s);
void     or_fwht_f32(float* x, int d);
/* the transform output channel the rotation stores at channel p (d = 128: the
 * 3-bit fields at bits 1-3 and 4-6 of p swapped; else p) */
int      or_rotation_channel(int p, int d);

/* ---- document bookkeeping ---- */
/* number of document-local blocks of `block` tokens: sum over documents of ceil(L/block) */
long     or_num_blocks(const int32_t* cu_seqlens, int num_docs, int total_tokens, int block);

/* ---- O-2 quantiser ----
 * x: [T][H][d] fp32 values (bf16 inputs widened exactly).
 * codes: [T][H][d] E4M3 bytes.
 * E4M3 token blocks : scales_f32 [H][NB], NB = or_num_blocks(.., block)
 * MX row32 (Q, K)   : scales_u8  [T][H][d/32] (biased E8M0 bytes)
 * MX col32 (V)      : scales_u8  [H][NG][d], NG = or_num_blocks(.., 32)
 * NVFP4 (Q, K)      : codes [T][H][d/2] (two E2M1 codes per byte, the even
 *                     channel in the low nibble); scales_f32 [H][NB] (fp32
 *                     scale per document-local 128-token block, block = 128);
 *                     scales_u8 [T][H][d/16] (E4M3 scale per 16 channels)
 */
int or_quantize(const float* x, int T, int H, int d, const int32_t* cu_seqlens, int num_docs,
                int layout, int block, int rotate, uint64_t seed, int mx_rule,
                uint8_t* codes, float* scales_f32, uint8_t* scales_u8);

/* ---- O-1 FP64 attention ----
 * rows: global token indices to evaluate (NULL => all T, in order).
 * o: [nrows][H][d], lse: [H][nrows] (natural log of the scaled scores).
 */
void or_attention_fp64(const double* q, const double* k, const double* v, int T, int H, int d,
                       const int32_t* cu_seqlens, int num_docs, int causal, double softmax_scale,
                       const int32_t* rows, int nrows, double* o, double* lse);

/* ---- O-1 backward: dQ, dK, dV of the FP64 attention for an upstream dO ----
 * All arrays [T][H][d] fp64; masking and documents as in or_attention_fp64.
 */
void or_attention_fp64_bwd(const double* q, const double* k, const double* v, const double* dout, int T, int H,
                           int d, const int32_t* cu_seqlens, int num_docs, int causal, double softmax_scale,
                           double* dq, double* dk, double* dv);
/* The same with D_i = dout_i . o_i taken from a given output o [T][H][d] (the
 * forward's stored output; NULL = or_attention_fp64_bwd). */
void or_attention_fp64_bwd_o(const double* q, const double* k, const double* v, const double* dout,
                             const double* o, int T, int H, int d, const int32_t* cu_seqlens, int num_docs,
                             int causal, double softmax_scale, double* dq, double* dk, double* dv);

/* ---- O-3 quantised-operand emulation ---- */
typedef struct {
    const uint8_t* codes;       /* [T][H][d] */
    int layout;                 /* OR_E4M3_TOKBLOCK / OR_MX_ROW32 / OR_MX_COL32 / OR_MX_TOKEN */
    int block;                  /* token block for OR_E4M3_TOKBLOCK */
    const float* scales_f32;    /* E4M3 layout */
    const uint8_t* scales_u8;   /* MX layouts */
} or_qtensor;

/* flags. The exponential of the probabilities (default: 2^x itself, the
 * hardware exp2's target): OR_EMU_EXP_SCHRAUDOLPH or OR_EMU_EXP_MITCHELL_P
 * select the bit-level forms below (with E4M3 P; E4M3 block-128 or MX col32
 * V; not causal-exact). */
enum { OR_EMU_QUANTIZE_P = 1, OR_EMU_EXP_SCHRAUDOLPH = 2, OR_EMU_EXP_MITCHELL_P = 4 };

/* ---- bit-level exponentials (FLAMIA sections 1, 4.3, 4.4) ----
 * Both take u = x - OR_SCHRAUDOLPH_DELTA, delta = log2(1/2 + 3 / (8 ln 2)).
 * or_exp2_schraudolph: 2^floor(u) (1 + frac(u)), u resolved to 2^-14 (to
 *   nearest, ties to even) and limited to u >= -126: the fp32 value whose
 *   bit pattern is 2^23 (u + 127) (Schraudolph's exponential).
 * or_exp2_mitchell_code: the E4M3 code round(8 u + 56) (ties to even),
 *   limited to [0, 126]: the code read as a fixed-point log2 (Mitchell). */
#define OR_SCHRAUDOLPH_DELTA 0.057984814725439975
float   or_exp2_schraudolph(double x);
uint8_t or_exp2_mitchell_code(double x);

/* rows as for O-1; o, o_bf16: [nrows][H][d]; lse: [H][nrows].
 * amb (NULL to skip): [nrows][H][d], the part of each output element that
 * E4M3 probability codes within rounding of a code boundary could move (the
 * tie allowance described beside the implementation).
 * lse_amb (NULL to skip): [H][nrows], the same for lse (natural log units):
 * non-zero only under the log-domain P, whose row sum adds the codes' values,
 * so that a tie there moves l as well: -ln(1 - Lt / l), Lt the sum over tied
 * keys of |code_hi - code_lo| / r, rescaled like l. */

int or_attention_emulate(const or_qtensor* q, const or_qtensor* k, const or_qtensor* v,
                         int T, int H, int d, const int32_t* cu_seqlens, int num_docs,
                         int causal, int exact, int rotated, double softmax_scale, float rescale_tau, int flags,
                         const int32_t* rows, int nrows, float* o, uint16_t* o_bf16, float* lse,
                         float* amb, float* lse_amb);

/* The emulation with a device's E4M3 probability codes checked and substituted
 * for its own: p_codes[(h * T + t) * p_stride + k] is the code row t of head h
 * gave document-local key k (0 for keys the row does not see). counts[4]:
 * keys with the emulation's own code, keys with the other faithful code of a
 * tie, keys with any other code, unseen keys with a non-zero code. */
int or_attention_emulate_given_p(const or_qtensor* q, const or_qtensor* k, const or_qtensor* v,
                                 int T, int H, int d, const int32_t* cu_seqlens, int num_docs,
                                 int causal, int exact, int rotated, double softmax_scale, float rescale_tau,
                                 int flags, const int32_t* rows, int nrows, float* o, uint16_t* o_bf16, float* lse,
                                 const uint8_t* p_codes, long p_stride, long* counts);

#ifdef __cplusplus
}
#endif
#endif
