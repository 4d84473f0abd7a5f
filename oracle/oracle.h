/*
 * oracle.h -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, float64 CPU oracle for the MLX-style group-affine quantized
 * linear projection.  It exists so that tests/ and the bench's CPU baseline
 * can check the CUDA library against an independent implementation.  Nothing
 * in the product path (the libaffqmm library and its Python binding) may
 * include, link or call this code, and this code includes nothing of theirs.
 *
 * Inputs are the canonical, unpacked form of an affine table:
 *   codes  q[N,K]   one code per byte, 0 <= q < 2^bits
 *   scales s[N,K/g] bf16 bit patterns (uint16), row-major
 *   biases b[N,K/g] bf16 bit patterns (uint16), row-major
 *   x[M,K]          bf16 bit patterns, row-major
 * Group j of row n covers k in [j*g, (j+1)*g).
 *
 * Sources (web pages on the TensorFold project):
 *  - "Gemma 4 12B on the native Metal engine" (PR #975), the commit that makes
 *    the prompt GEMM dequantize each weight as bf16(fma(scale, code, bias)) with
 *    one rounding, as mlx-lm's quantized matmul does, and accumulate over the
 *    whole depth; the same page's lane kernels that keep codes exact and use
 *    precomputed group sums (the commit on the reg variant of the lane kernel).
 *  - "cuda gemma4: images on the 12B ..." (PR #1183), the embed_rows commit
 *    (MLX affine tables at 2/3/4/5/6/8 bits, groups of 32/64/128) and the
 *    bf16 rounding commit (signed zero from underflow, subnormal ties, the
 *    normal boundary, overflow to both infinities).
 *
 * Every function returns 0 on success and a negative value on a bad argument.
 */
#ifndef GAB_ORACLE_H
#define GAB_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* bf16 round-to-nearest-even of a double: NaN stays NaN (0x7FC0, sign kept),
 * overflow gives +-inf, underflow keeps the sign (-2^-135 -> 0x8000). */
uint16_t oracle_bf16_from_double(double v);
/* The exact value of a bf16 bit pattern. */
double oracle_bf16_to_double(uint16_t h);
/* Encode n fp32 bit patterns (as uint32) to bf16 through the double path. */
void oracle_bf16_from_f32_bits(const uint32_t* in, uint16_t* out, size_t n);

/* One weight: bf16(s*q + b) with a single rounding of the exact value. */
uint16_t oracle_dequant_one(uint32_t q, uint16_t s, uint16_t b);

/* W[n,k] = bf16(s[n,k/g]*q[n,k] + b[n,k/g]), all N*K weights. */
int oracle_dequant(int bits, int group, int64_t N, int64_t K,
                   const uint8_t* codes, const uint16_t* scales,
                   const uint16_t* biases, uint16_t* w_out);

/* y[m,n] = sum over k ascending of W[n,k]*x[m,k], in double.
 * y_out is [M,N] row-major.  nthreads <= 1 runs on the calling thread;
 * otherwise output rows n are split into nthreads contiguous ranges. */
int oracle_qmm(int bits, int group, int64_t M, int64_t N, int64_t K,
               const uint16_t* x, const uint8_t* codes,
               const uint16_t* scales, const uint16_t* biases,
               double* y_out, int nthreads);

/* The exact-codes form used by the pages' lane kernels:
 * y_gs[m,n] = sum_j ( s_j * sum_{k in j} q[n,k]*x[m,k] + b_j * sum_{k in j} x[m,k] ),
 * in double, with no bf16 rounding of the weights.  Also writes
 * mag[m,n] = sum_k |s*q + b| * |x[m,k]| (exact weights, double), the scale the
 * group-sum invariant is stated against.  Either output pointer may be NULL. */
int oracle_qmm_groupsum(int bits, int group, int64_t M, int64_t N, int64_t K,
                        const uint16_t* x, const uint8_t* codes,
                        const uint16_t* scales, const uint16_t* biases,
                        double* y_gs, double* mag);

/* The exact-codes form with the group sums of x supplied by the caller, as
 * the kernel that produced x writes them ("Gemma 4 12B on the native Metal
 * engine" page, the commit where the norm, merge, attention-tail, geglu and
 * dense-tail kernels write the next projection's group sums):
 * y[m,n] = sum_j ( s_j * sum_{k in j} q[n,k]*x[m,k] + b_j * xsums[m,j] ),
 * in double; xsums is fp32 [M, K/g] and is used as given. */
int oracle_qmm_groupsum_given(int bits, int group, int64_t M, int64_t N, int64_t K,
                              const uint16_t* x, const float* xsums, const uint8_t* codes,
                              const uint16_t* scales, const uint16_t* biases, double* y);

/* mlx_lm's GeGLU on bf16 rows, h = gelu_approx(gate) * up, as MLX evaluates it
 * on bf16 arrays: every operation's exact result rounded once to bf16, the
 * constants taken as bf16:
 *   c3 = bf16(g^3)        c1 = bf16(0.044715)     a = bf16(c1 * c3)
 *   z  = bf16(g + a)      c2 = bf16(sqrt(2/pi))   u = bf16(c2 * z)
 *   t  = bf16(tanh(u))    e  = bf16(1 + t)        p = bf16(0.5 * g)
 *   r  = bf16(p * e)      h  = bf16(r * up)
 * ("cuda gemma4" page: tf_geglu_rows computes mlx_lm's gelu_approx(gate) * up
 * as MLX's bf16 ops; "Gemma 4 12B on the native Metal engine" page: geglu as
 * the gate/up projection's epilogue, its results equal to the unfused ones).  tanh is the
 * double library function.  A GPU's fp32 tanh is within `tanh_ulps` fp32
 * ulps of the exact value, so where the exact tanh lies that close to a bf16
 * rounding boundary the bf16 t has two possible values: h_lo takes the one
 * below, h_hi the one above (equal everywhere else).  NaN and infinities
 * propagate as IEEE arithmetic does. */
void oracle_geglu(int64_t n, const uint16_t* gate, const uint16_t* up, int tanh_ulps,
                  uint16_t* h_lo, uint16_t* h_hi);

/* Scaled embedding rows: out[t,k] = bf16( bf16(s*q + b) * scale ) for the
 * table row n = ids[t] -- two roundings, each of an exact value: the weight
 * (as oracle_dequant_one) and then its exact product with the bf16 scale.
 * "cuda gemma4: images on the 12B" page, the embed_rows commit.  has_scale = 0
 * gives the weight row itself (no second rounding).  out is [T,K] row-major.
 * Returns -6 if an id is outside [0, N). */
int oracle_embed_rows(int bits, int group, int64_t N, int64_t K,
                      const uint8_t* codes, const uint16_t* scales,
                      const uint16_t* biases, const int32_t* ids, int64_t T,
                      int has_scale, uint16_t scale, uint16_t* out);

#ifdef __cplusplus
}
#endif
#endif
