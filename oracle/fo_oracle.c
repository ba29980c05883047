/*
 * fo_oracle.c -- plain CPU oracle of the FlashAdamW step (TEST INFRASTRUCTURE).
 *
 * Only the test-suite, the smoke check and the benchmark's CPU baseline call
 * this file.  It is deliberately slow and literal: one full pass over the
 * tensor per line of the pages' code, every operation a separately rounded
 * binary32 operation.  See fo_oracle.h for the sources.
 *
 * Pinning status (what each function is checked against, in the CPU tests):
 *   f32<->f16, f32->bf16   torch's own conversions, exhaustively / on sweeps.
 *   quantize/dequantize    hand-worked single groups, numpy float16 scales,
 *                          sign and power-of-two invariances, brute-force
 *                          nearest-code search in binary64, error bounds,
 *                          padding identity.
 *   split/reconstruct      all 2^32 inputs (32-bit master exact), an
 *                          independent binary64 rounding of the 24-bit master,
 *                          torch's bf16 rounding away from ties.
 *   adamw_step             torch.optim.AdamW (float64) for the unquantized
 *                          fp32 special case, first-step closed form from
 *                          zero state, a multi-step closed form for
 *                          constant-gradient groups, zero-grad invariants.
 *                          Beyond these the multi-step trajectory on random
 *                          data rests on the definition itself.
 */
#include "fo_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#define GROUP 32

static uint32_t bits_of(float f) {
  uint32_t b;
  memcpy(&b, &f, 4);
  return b;
}
static float float_of(uint32_t b) {
  float f;
  memcpy(&f, &b, 4);
  return f;
}

/* ------------------------------------------------------------------------ */
/* Number formats                                                           */
/* ------------------------------------------------------------------------ */

/* Round the non-negative integer `v` right by `s` bits, to nearest, ties to
 * even.  1 <= s <= 31. */
static uint32_t shift_right_rne(uint32_t v, int s) {
  uint32_t q = v >> s;
  uint32_t rem = v & ((1u << s) - 1u);
  uint32_t half = 1u << (s - 1);
  if (rem > half || (rem == half && (q & 1u))) q += 1u;
  return q;
}

uint16_t fo_oracle_f32_to_f16(float f) {
  uint32_t x = bits_of(f);
  uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
  uint32_t exp = (x >> 23) & 0xFFu;
  uint32_t man = x & 0x7FFFFFu;
  if (exp == 0xFFu) {                      /* inf or NaN */
    if (man == 0) return (uint16_t)(sign | 0x7C00u);
    return (uint16_t)(sign | 0x7E00u | (man >> 13));
  }
  if (exp == 0) return sign;               /* fp32 subnormal or zero: far below half's range */
  int e = (int)exp - 127;                  /* value = 1.man * 2^e */
  uint32_t full = (1u << 23) | man;        /* 24-bit significand */
  if (e > 15) return (uint16_t)(sign | 0x7C00u);
  if (e >= -14) {
    /* normal half: keep 10 fraction bits; a carry out of the fraction bumps
     * the exponent, and out of e = 15 gives 0x7C00 = infinity. */
    uint32_t q = shift_right_rne(full, 13); /* 11-bit significand incl. hidden bit (or 2^11 on carry) */
    uint32_t h = ((uint32_t)(e + 15) << 10) + (q - (1u << 10));
    return (uint16_t)(sign | h);
  }
  /* subnormal half: count units of 2^-24; value / 2^-24 = full * 2^(e+1). */
  int s = -(e + 1);                         /* >= 14 */
  if (s > 24) return sign;                  /* below 2^-25: rounds to zero */
  uint32_t q = shift_right_rne(full, s);    /* may reach 0x400 = smallest normal: still the right code */
  return (uint16_t)(sign | q);
}

float fo_oracle_f16_to_f32(uint16_t h) {
  uint32_t sign = ((uint32_t)h & 0x8000u) << 16;
  uint32_t exp = ((uint32_t)h >> 10) & 0x1Fu;
  uint32_t man = (uint32_t)h & 0x3FFu;
  if (exp == 0) {
    float mag = ldexpf((float)man, -24);    /* exact: man < 2^10 */
    return sign ? -mag : mag;
  }
  if (exp == 31) return float_of(sign | 0x7F800000u | (man << 13));
  return float_of(sign | ((exp - 15u + 127u) << 23) | (man << 13));
}

uint16_t fo_oracle_f32_to_bf16_rne(float f) {
  uint32_t x = bits_of(f);
  if ((x & 0x7F800000u) == 0x7F800000u && (x & 0x7FFFFFu)) /* NaN: keep it quiet */
    return (uint16_t)((x >> 16) | 0x40u);
  uint32_t sign = x & 0x80000000u;
  uint32_t mag = x & 0x7FFFFFFFu;
  uint32_t q = shift_right_rne(mag, 16);    /* magnitude in bf16 units; overflow lands on inf */
  return (uint16_t)((sign >> 16) | q);
}

void fo_oracle_f32_to_f16_array(const float* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = fo_oracle_f32_to_f16(x[i]);
}
void fo_oracle_f16_to_f32_array(const uint16_t* h, int64_t n, float* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = fo_oracle_f16_to_f32(h[i]);
}
void fo_oracle_f32_to_bf16_rne_array(const float* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = fo_oracle_f32_to_bf16_rne(x[i]);
}

/* ------------------------------------------------------------------------ */
/* [Q] quantize / dequantize                                                */
/* ------------------------------------------------------------------------ */

/* Page "code/flashsim/quantization.py", `quantize`: the input is cut into
 * groups of 32 after zero padding (`_grouped`); optional square root; the
 * group scale is the max of |x| (signed) or of x (unsigned), rounded to fp16;
 * a zero fp16 scale is replaced by 1 for the division only; optional softsign
 * 2y/(1+|y|); codes are round-half-even of 127y clamped to [-127,127]
 * (int8) or of 255y clamped to [0,255] (uint8); codes are kept for the first
 * n elements and every group's fp16 scale is returned. */
void fo_oracle_quantize(const float* x, int64_t n, int is_signed, int use_sqrt, int use_softsign,
                        void* codes, uint16_t* scales) {
  int64_t n_groups = (n + GROUP - 1) / GROUP;
  for (int64_t gi = 0; gi < n_groups; ++gi) {
    float g[GROUP];
    for (int j = 0; j < GROUP; ++j) {
      int64_t idx = gi * GROUP + j;
      g[j] = idx < n ? x[idx] : 0.0f;       /* `_grouped`: pad with zeros */
    }
    if (use_sqrt)
      for (int j = 0; j < GROUP; ++j) g[j] = sqrtf(g[j]);

    float a = is_signed ? fabsf(g[0]) : g[0];
    for (int j = 1; j < GROUP; ++j) {
      float c = is_signed ? fabsf(g[j]) : g[j];
      if (c > a) a = c;
    }
    uint16_t s16 = fo_oracle_f32_to_f16(a);
    float s_f = fo_oracle_f16_to_f32(s16);
    float safe = (s_f == 0.0f) ? 1.0f : s_f;

    for (int j = 0; j < GROUP; ++j) {
      int64_t idx = gi * GROUP + j;
      float y = g[j] / safe;
      if (use_softsign) y = (2.0f * y) / (1.0f + fabsf(y));
      if (is_signed) {
        float t = rintf(y * 127.0f);
        if (t < -127.0f) t = -127.0f;
        if (t > 127.0f) t = 127.0f;
        if (idx < n) ((int8_t*)codes)[idx] = (int8_t)t;
      } else {
        float t = rintf(y * 255.0f);
        if (t < 0.0f) t = 0.0f;
        if (t > 255.0f) t = 255.0f;
        if (idx < n) ((uint8_t*)codes)[idx] = (uint8_t)t;
      }
    }
    scales[gi] = s16;
  }
}

/* Page "code/flashsim/quantization.py", `dequantize`: y = code/127 (signed) or
 * code/255 (unsigned); optional inverse softsign y/(2-|y|); times the stored
 * fp16 scale (not the zero-guarded one); optional square. */
void fo_oracle_dequantize(const void* codes, const uint16_t* scales, int64_t n, int is_signed,
                          int use_sqrt, int use_softsign, float* out) {
  for (int64_t i = 0; i < n; ++i) {
    float s = fo_oracle_f16_to_f32(scales[i / GROUP]);
    float q = is_signed ? (float)((const int8_t*)codes)[i] : (float)((const uint8_t*)codes)[i];
    float y = q / (is_signed ? 127.0f : 255.0f);
    if (use_softsign) y = y / (2.0f - fabsf(y));
    float o = y * s;
    if (use_sqrt) o = o * o;
    out[i] = o;
  }
}

/* ------------------------------------------------------------------------ */
/* [H] split / reconstruct                                                  */
/* ------------------------------------------------------------------------ */

/* The pages call the pair (compute_ecc_bits / reconstruct_fp32_param, or the
 * simulator's compress / decompress) with a 3- or 4-byte master weight but do
 * not print their source.  Reading taken here:
 *   1. the master weight is theta rounded to an M-bit float (M = 24 or 32:
 *      sign, 8 exponent bits, M-9 fraction bits), to nearest, ties away from
 *      zero -- on the bit pattern, add half of the dropped unit to the
 *      magnitude bits and truncate;
 *   2. the bf16 parameter theta' is that master rounded the same way to 16
 *      bits;
 *   3. rho is the exact difference master - theta'<<16 in units of the
 *      master's last place; it always fits int8 (M = 24) or int16 (M = 32);
 *   4. reconstruction adds theta'<<16 and rho<<(32-M) as integers, giving the
 *      master back bit for bit.
 * NaN splits to a quiet bf16 NaN of the same sign with rho = 0. */
static int master_shift(int master_bits) {
  if (master_bits == 24) return 8;
  if (master_bits == 32) return 0;
  return -1;
}

int fo_oracle_split(const float* theta, int64_t n, int master_bits, uint16_t* theta_bf16, void* rho) {
  int sh = master_shift(master_bits);
  if (sh < 0) return -1;
  for (int64_t i = 0; i < n; ++i) {
    uint32_t b = bits_of(theta[i]);
    int32_t r;
    uint16_t hi;
    if ((b & 0x7F800000u) == 0x7F800000u && (b & 0x7FFFFFu)) {
      hi = (uint16_t)(((b >> 16) & 0x8000u) | 0x7FC0u);
      r = 0;
    } else {
      uint32_t master = b;
      if (sh) master = (b + (1u << (sh - 1))) & ~((1u << sh) - 1u);
      hi = (uint16_t)((master + 0x8000u) >> 16);
      int32_t diff = (int32_t)(master - ((uint32_t)hi << 16));
      r = diff / (1 << sh);                 /* exact: diff is a multiple of 2^sh */
    }
    theta_bf16[i] = hi;
    if (sh) ((int8_t*)rho)[i] = (int8_t)r;
    else ((int16_t*)rho)[i] = (int16_t)r;
  }
  return 0;
}

int fo_oracle_reconstruct(const uint16_t* theta_bf16, const void* rho, int64_t n, int master_bits,
                          float* theta) {
  int sh = master_shift(master_bits);
  if (sh < 0) return -1;
  for (int64_t i = 0; i < n; ++i) {
    int32_t r = sh ? (int32_t)((const int8_t*)rho)[i] : (int32_t)((const int16_t*)rho)[i];
    uint32_t b = ((uint32_t)theta_bf16[i] << 16) + (uint32_t)(r * (1 << sh));
    theta[i] = float_of(b);
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* [A] one FlashAdamW step on one tensor                                    */
/* ------------------------------------------------------------------------ */

/* Page "code/flashsim/flash_adamw_sim.py", `FlashAdamWSim.step`, for one
 * parameter whose state already exists:
 *   g = grad as fp32
 *   prologue: m = dequantize(m), v = dequantize(v), theta = reconstruct(theta', rho)
 *   if wd != 0: theta = theta * (1 - lr*wd)
 *   m = beta1*m + (1-beta1)*g
 *   v = beta2*v + (1-beta2)*g*g            (evaluated left to right)
 *   mhat = m / (1 - beta1^t);  vhat = v / (1 - beta2^t)
 *   theta = theta - lr*mhat / (sqrt(vhat) + eps)
 *   epilogue: m, v re-quantized with fresh scales; theta re-split.
 * Momentum uses the signed softsign spec, variance the unsigned sqrt spec
 * (both linear when companded = 0).  Each line is a full pass, as in the
 * simulator. */
int fo_oracle_adamw_step(int64_t n, void* param, int param_kind, void* rho, const void* grad,
                         int grad_kind, void* m_state, uint16_t* m_scales, void* v_state,
                         uint16_t* v_scales, int quantize_states, int companded, double lr,
                         double beta1, double beta2, double eps, double weight_decay, int64_t step) {
  if (n < 0 || step < 1) return -1;
  if (param_kind < 0 || param_kind > 3 || (grad_kind != 0 && grad_kind != 1)) return -1;
  if (n == 0) return 0;
  size_t bytes = (size_t)n * sizeof(float);
  float* g = (float*)malloc(bytes);
  float* m = (float*)malloc(bytes);
  float* v = (float*)malloc(bytes);
  float* theta = (float*)malloc(bytes);
  if (!g || !m || !v || !theta) {
    free(g); free(m); free(v); free(theta);
    return -1;
  }

  /* g = p.grad.float() */
  for (int64_t i = 0; i < n; ++i) {
    if (grad_kind == FO_ORACLE_GRAD_F32) g[i] = ((const float*)grad)[i];
    else g[i] = float_of((uint32_t)((const uint16_t*)grad)[i] << 16);
  }

  /* prologue */
  int m_sqrt = 0, m_soft = companded ? 1 : 0;
  int v_sqrt = companded ? 1 : 0, v_soft = 0;
  if (quantize_states) {
    fo_oracle_dequantize(m_state, m_scales, n, 1, m_sqrt, m_soft, m);
    fo_oracle_dequantize(v_state, v_scales, n, 0, v_sqrt, v_soft, v);
  } else {
    memcpy(m, m_state, bytes);
    memcpy(v, v_state, bytes);
  }
  if (param_kind == FO_ORACLE_PARAM_BF16_RHO8 || param_kind == FO_ORACLE_PARAM_BF16_RHO16) {
    fo_oracle_reconstruct((const uint16_t*)param, rho, n,
                          param_kind == FO_ORACLE_PARAM_BF16_RHO8 ? 24 : 32, theta);
  } else if (param_kind == FO_ORACLE_PARAM_BF16) {
    for (int64_t i = 0; i < n; ++i) theta[i] = float_of((uint32_t)((uint16_t*)param)[i] << 16);
  } else {
    memcpy(theta, param, bytes);
  }

  /* Python-float scalars, rounded once to binary32 */
  const float c_wd = (float)(1.0 - lr * weight_decay);
  const float b1 = (float)beta1, one_minus_b1 = (float)(1.0 - beta1);
  const float b2 = (float)beta2, one_minus_b2 = (float)(1.0 - beta2);
  const float bc1 = (float)(1.0 - pow(beta1, (double)step));
  const float bc2 = (float)(1.0 - pow(beta2, (double)step));
  const float lr_f = (float)lr, eps_f = (float)eps;

  /* standard AdamW update, decoupled weight decay first */
  if (weight_decay != 0.0)
    for (int64_t i = 0; i < n; ++i) theta[i] = theta[i] * c_wd;
  for (int64_t i = 0; i < n; ++i) m[i] = b1 * m[i] + one_minus_b1 * g[i];
  for (int64_t i = 0; i < n; ++i) v[i] = b2 * v[i] + (one_minus_b2 * g[i]) * g[i];
  for (int64_t i = 0; i < n; ++i) {
    float mhat = m[i] / bc1;
    float vhat = v[i] / bc2;
    float num = lr_f * mhat;
    float den = sqrtf(vhat) + eps_f;
    theta[i] = theta[i] - num / den;
  }

  /* epilogue */
  if (quantize_states) {
    fo_oracle_quantize(m, n, 1, m_sqrt, m_soft, m_state, m_scales);
    fo_oracle_quantize(v, n, 0, v_sqrt, v_soft, v_state, v_scales);
  } else {
    memcpy(m_state, m, bytes);
    memcpy(v_state, v, bytes);
  }
  if (param_kind == FO_ORACLE_PARAM_BF16_RHO8 || param_kind == FO_ORACLE_PARAM_BF16_RHO16) {
    fo_oracle_split(theta, n, param_kind == FO_ORACLE_PARAM_BF16_RHO8 ? 24 : 32, (uint16_t*)param, rho);
  } else if (param_kind == FO_ORACLE_PARAM_BF16) {
    fo_oracle_f32_to_bf16_rne_array(theta, n, (uint16_t*)param);
  } else {
    memcpy(param, theta, bytes);
  }
  free(g); free(m); free(v); free(theta);
  return 0;
}

/* One FlashSGD step (the reading stated in fo_oracle.h [B]). */
int fo_oracle_sgd_step(int64_t n, void* param, int param_kind, void* rho, const void* grad, int grad_kind,
                       void* m_state, uint16_t* m_scales, int quantize_states, int companded, double lr,
                       double momentum, double weight_decay) {
  if (n < 0) return -1;
  if (param_kind < 0 || param_kind > 3 || (grad_kind != 0 && grad_kind != 1)) return -1;
  if (n == 0) return 0;
  size_t bytes = (size_t)n * sizeof(float);
  float* g = (float*)malloc(bytes);
  float* buf = (float*)malloc(bytes);
  float* theta = (float*)malloc(bytes);
  if (!g || !buf || !theta) {
    free(g); free(buf); free(theta);
    return -1;
  }
  for (int64_t i = 0; i < n; ++i) {
    if (grad_kind == FO_ORACLE_GRAD_F32) g[i] = ((const float*)grad)[i];
    else g[i] = float_of((uint32_t)((const uint16_t*)grad)[i] << 16);
  }
  /* prologue: the momentum buffer and the master weight */
  if (quantize_states) fo_oracle_dequantize(m_state, m_scales, n, 1, 0, companded ? 1 : 0, buf);
  else memcpy(buf, m_state, bytes);
  if (param_kind == FO_ORACLE_PARAM_BF16_RHO8 || param_kind == FO_ORACLE_PARAM_BF16_RHO16) {
    fo_oracle_reconstruct((const uint16_t*)param, rho, n, param_kind == FO_ORACLE_PARAM_BF16_RHO8 ? 24 : 32, theta);
  } else if (param_kind == FO_ORACLE_PARAM_BF16) {
    for (int64_t i = 0; i < n; ++i) theta[i] = float_of((uint32_t)((uint16_t*)param)[i] << 16);
  } else {
    memcpy(theta, param, bytes);
  }
  /* Python-float scalars, rounded once to binary32 */
  const float lr_f = (float)lr, mu = (float)momentum, wd = (float)weight_decay;
  for (int64_t i = 0; i < n; ++i) {
    float gi = g[i];
    if (weight_decay != 0.0) gi = gi + wd * theta[i];
    buf[i] = mu * buf[i] + gi;
    theta[i] = theta[i] - lr_f * buf[i];
  }
  /* epilogue */
  if (quantize_states) fo_oracle_quantize(buf, n, 1, 0, companded ? 1 : 0, m_state, m_scales);
  else memcpy(m_state, buf, bytes);
  if (param_kind == FO_ORACLE_PARAM_BF16_RHO8 || param_kind == FO_ORACLE_PARAM_BF16_RHO16) {
    fo_oracle_split(theta, n, param_kind == FO_ORACLE_PARAM_BF16_RHO8 ? 24 : 32, (uint16_t*)param, rho);
  } else if (param_kind == FO_ORACLE_PARAM_BF16) {
    fo_oracle_f32_to_bf16_rne_array(theta, n, (uint16_t*)param);
  } else {
    memcpy(param, theta, bytes);
  }
  free(g); free(buf); free(theta);
  return 0;
}
