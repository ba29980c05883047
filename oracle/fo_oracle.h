/*
 * fo_oracle.h -- plain CPU oracle of the FlashAdamW step and its kernel pairs.
 *
 * TEST INFRASTRUCTURE.  Only the test-suite, the smoke check and the CPU
 * baseline of the benchmark may call this code.  It shares nothing with the
 * CUDA library (no header, no helper, no table): it is a second, independent
 * statement of the same definitions, written to be read against the pages.
 *
 * Sources (page title, then the part of it that each function follows):
 *   [Q]  "code/flashsim/quantization.py": the module docstring (group-32
 *        companded quantization, Algorithms 2-3 of the FlashOptim paper),
 *        `_grouped`, `quantize`, `dequantize`.
 *   [A]  "code/flashsim/flash_adamw_sim.py": `FlashAdamWSim.step`
 *        (Algorithm 4: prologue, AdamW update, epilogue).
 *   [H]  "code/gpu/equivalence.py": `eq_ecc` (how the split pair is called:
 *        compute_ecc_bits / reconstruct_fp32_param with a 3- or 4-byte master).
 *
 * All arithmetic is IEEE binary32 with round-to-nearest-even, one rounding per
 * operation (built with -ffp-contract=off, no fast-math), in the order the
 * pages write it.  Python float scalars are formed in binary64 and rounded to
 * binary32 once, as torch does when it multiplies an fp32 tensor by a Python
 * float.
 */
#ifndef FO_ORACLE_H
#define FO_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- number formats ----------------------------------------------------- */
/* binary32 -> binary16, round to nearest even; subnormal results kept; values
 * at or above 65520 in magnitude become infinity (torch `Tensor.half()`). */
uint16_t fo_oracle_f32_to_f16(float f);
float fo_oracle_f16_to_f32(uint16_t h);
/* binary32 -> bfloat16, round to nearest even (torch `.to(torch.bfloat16)`). */
uint16_t fo_oracle_f32_to_bf16_rne(float f);

void fo_oracle_f32_to_f16_array(const float* x, int64_t n, uint16_t* out);
void fo_oracle_f16_to_f32_array(const uint16_t* h, int64_t n, float* out);
void fo_oracle_f32_to_bf16_rne_array(const float* x, int64_t n, uint16_t* out);

/* ---- [Q] group-32 quantize / dequantize --------------------------------- */
/* x[n] fp32 -> codes[n] (int8 if is_signed else uint8) and fp16 scales
 * [ceil(n/32)] (raw binary16 bits).  Momentum = (1,0,1); variance = (0,1,0);
 * the linear ablations are (1,0,0) and (0,0,0). */
void fo_oracle_quantize(const float* x, int64_t n, int is_signed, int use_sqrt, int use_softsign,
                        void* codes, uint16_t* scales);
void fo_oracle_dequantize(const void* codes, const uint16_t* scales, int64_t n, int is_signed,
                          int use_sqrt, int use_softsign, float* out);

/* ---- [H] split / reconstruct (24- or 32-bit master) --------------------- */
/* master_bits = 24 (rho int8) or 32 (rho int16).  Returns 0, or -1 on a bad
 * master_bits. */
int fo_oracle_split(const float* theta, int64_t n, int master_bits, uint16_t* theta_bf16, void* rho);
int fo_oracle_reconstruct(const uint16_t* theta_bf16, const void* rho, int64_t n, int master_bits,
                          float* theta);

/* ---- [A] one FlashAdamW step on one tensor ------------------------------ */
enum {
  FO_ORACLE_PARAM_BF16_RHO8 = 0,  /* master_weight_bits = 24 */
  FO_ORACLE_PARAM_BF16_RHO16 = 1, /* master_weight_bits = 32 */
  FO_ORACLE_PARAM_BF16 = 2,       /* master_weight_bits = None, bf16 parameter */
  FO_ORACLE_PARAM_F32 = 3         /* fp32 parameter: no split */
};
enum { FO_ORACLE_GRAD_F32 = 0, FO_ORACLE_GRAD_BF16 = 1 };

/* In place on param / rho / m / v.  With quantize_states = 1, m_state is
 * int8[n] + m_scales fp16[ceil(n/32)] and v_state uint8[n] + v_scales; with
 * quantize_states = 0 they are fp32[n] and the scale pointers are unused.
 * companded = 0 selects the linear ablation for both states.  `step` is the
 * already-incremented step count t >= 1.  Returns 0, or -1 on bad arguments
 * or allocation failure. */
int fo_oracle_adamw_step(int64_t n, void* param, int param_kind, void* rho, const void* grad,
                         int grad_kind, void* m_state, uint16_t* m_scales, void* v_state,
                         uint16_t* v_scales, int quantize_states, int companded, double lr,
                         double beta1, double beta2, double eps, double weight_decay, int64_t step);

/* ---- [B] one FlashSGD step on one tensor ------------------------------- */
/* The pages name FlashSGD only in the byte accounting of
 * "code/flashsim/flash_adamw_sim.py" (`bytes_per_param`: the master weight
 * split as in FlashAdamW and one quantized state, the momentum).  The update
 * read here is SGD with momentum as in torch.optim.SGD (dampening 0, no
 * Nesterov, weight decay added to the gradient), every operation rounded
 * once:
 *   g = fp32(grad); if wd != 0: g = g + wd * theta;
 *   buf = momentum * buf + g;  theta = theta - lr * buf
 * with buf stored like FlashAdamW's m (MOMENTUM spec, or MOMENTUM_LINEAR with
 * companded = 0, or fp32 with quantize_states = 0).  A zero buffer makes the
 * first step buf = g, as torch's clone of the first gradient does.  Same
 * parameter kinds and return values as fo_oracle_adamw_step. */
int fo_oracle_sgd_step(int64_t n, void* param, int param_kind, void* rho, const void* grad, int grad_kind,
                       void* m_state, uint16_t* m_scales, int quantize_states, int companded, double lr,
                       double momentum, double weight_decay);

#ifdef __cplusplus
}
#endif
#endif
