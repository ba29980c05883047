/*
 * fo.h -- C ABI of the GB300 FlashAdamW library (libfo.so).
 *
 * FlashAdamW keeps AdamW's optimizer state in 8 bits per value and the fp32
 * master weight as a bf16 parameter plus a small integer residual:
 *   - momentum m: int8 codes, one fp16 scale per group of 32, softsign
 *     companding (Alg. 2);
 *   - variance v: uint8 codes, one fp16 scale per group of 32, stored in the
 *     square-root domain (Alg. 3);
 *   - master weight: bf16 theta' plus rho, int8 (24-bit master) or int16
 *     (32-bit master).
 * Sources: the pages "code/flashsim/quantization.py" (module docstring,
 * `quantize`, `dequantize`), "code/flashsim/flash_adamw_sim.py"
 * (`FlashAdamWSim.step`, Algorithm 4) and "code/gpu/equivalence.py" (`eq_ecc`:
 * compute_ecc_bits / reconstruct_fp32_param with a 3- or 4-byte master).
 *
 * Conventions shared by every entry point:
 *   - All data pointers are DEVICE pointers (memory the GPU can address; the
 *     caller allocates and owns it, e.g. through torch).  The library
 *     allocates no device memory and never synchronizes the stream.
 *   - Element arrays must start on a 16-byte boundary, and so must the fp16
 *     scale arrays; otherwise FO_ERR_MISALIGNED is returned.
 *   - n (numel) may be any value >= 0; n = 0 is a no-op returning FO_OK.
 *     Scale arrays hold ceil(n/32) entries; a last group with fewer than 32
 *     live elements is quantized as if zero-padded (`_grouped`), and codes
 *     are written for the n live elements only.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Work is enqueued asynchronously; a launch failure is reported
 *     as FO_ERR_CUDA, and faults during execution surface at the caller's
 *     next synchronization, as with any stream API.
 *   - Argument errors return before any CUDA call is made.
 *   - Inputs are assumed finite.  Variance-spec inputs must be >= 0 (pass |x|
 *     or v); a negative input yields NaN from the square root, as in the
 *     reference.
 *   - Results are bit-identical to the binary32 definitions on the pages
 *     (IEEE division, square root and round-half-even; no FMA contraction).
 */
#ifndef FO_H
#define FO_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FO_OK = 0,
  FO_ERR_INVALID_ARG = 1, /* null pointer with n > 0, n < 0, bad enum, bad hyper-parameter */
  FO_ERR_MISALIGNED = 2,  /* a pointer not on a 16-byte boundary */
  FO_ERR_CUDA = 3,        /* the CUDA runtime refused a launch; see fo_last_cuda_error() */
  FO_ERR_ALIAS = 4,       /* fo_adamw_step: a written buffer overlaps another buffer */
  FO_ERR_TOO_LARGE = 5    /* fo_adamw_step_static: more tensors than FO_STATIC_MAX_TENSORS */
} fo_status;

/* Quantization spec of a state tensor.  MOMENTUM: signed int8, softsign
 * companding (Alg. 2).  VARIANCE: unsigned uint8, square root before
 * quantization and square after dequantization (Alg. 3).  The *_LINEAR specs
 * are the non-companded ablation of the quantization page (`momentum_linear`,
 * `variance_linear`): plain group absmax, no softsign, no square root. */
typedef enum {
  FO_SPEC_MOMENTUM = 0,
  FO_SPEC_VARIANCE = 1,
  FO_SPEC_MOMENTUM_LINEAR = 2,
  FO_SPEC_VARIANCE_LINEAR = 3
} fo_spec;

typedef enum { FO_DT_F32 = 0, FO_DT_BF16 = 1 } fo_dtype;

/* Human-readable name of a status code (static string). */
const char* fo_status_string(fo_status s);
/* Text of the last CUDA error seen by this thread's calls ("" if none). */
const char* fo_last_cuda_error(void);

/* ---- quantize / dequantize pair ------------------------------------------
 * "code/flashsim/quantization.py", `quantize`: x[n] fp32 -> codes[n]
 * (int8 for the signed specs, uint8 for the unsigned ones) and scales
 * [ceil(n/32)] (IEEE binary16 bits).  Per group of 32: optional sqrt; scale
 * = fp16(max |x|) (signed) or fp16(max x) (unsigned), round to nearest even,
 * overflow to +inf; a zero scale divides by 1 instead; optional softsign
 * 2y/(1+|y|); code = round-half-even(127 y) clamped to [-127, 127], or
 * round-half-even(255 y) clamped to [0, 255].  x is read-only; codes and
 * scales are written. */
fo_status fo_quantize(const float* x, int64_t n, fo_spec spec, void* codes, uint16_t* scales,
                      void* stream);

/* "code/flashsim/quantization.py", `dequantize`: codes[n] + scales -> out[n]
 * fp32.  y = code/127 (signed) or code/255 (unsigned); MOMENTUM applies the
 * inverse softsign y/(2-|y|); out = y * scale (the stored fp16 value, so a
 * zero scale gives 0 and an infinite one gives NaN for code 0); VARIANCE
 * squares the result. */
fo_status fo_dequantize(const void* codes, const uint16_t* scales, int64_t n, fo_spec spec,
                        float* out, void* stream);

/* ---- split / reconstruct pair ---------------------------------------------
 * "code/gpu/equivalence.py", `eq_ecc` (compute_ecc_bits with a 3- or 4-byte
 * master).  The pages do not print the rule; this library uses: the master
 * weight is theta rounded to a (8 + rho_bits + 16)-bit float -- 24 bits for
 * rho_bits = 8, 32 bits (= theta itself) for rho_bits = 16 -- to nearest,
 * ties away from zero; theta' (bf16 bits) is the master rounded the same way
 * to 16 bits; rho (int8 or int16) is the exact residual master - theta' in
 * units of the master's last place.  Reconstruction returns the master bit
 * for bit: exact fp32 for rho_bits = 16, within 2^-16 relative for 8.  NaN
 * splits to a quiet bf16 NaN with rho = 0.  theta is read-only. */
fo_status fo_split(const float* theta, int64_t n, int rho_bits, uint16_t* theta_bf16, void* rho,
                   void* stream);
/* reconstruct_fp32_param: bits(theta) = (theta' << 16) + (rho << (16 - rho_bits)). */
fo_status fo_reconstruct(const uint16_t* theta_bf16, const void* rho, int64_t n, int rho_bits,
                         float* theta, void* stream);

/* ---- fused multi-tensor FlashAdamW step -----------------------------------
 * One parameter tensor's buffers.  All are device pointers, updated in place
 * except `grad`:
 *   param    bf16 theta' bits [numel]
 *   rho      int8 or int16 [numel] (width = rho_bits of the call)
 *   grad     fp32 or bf16 [numel] (dtype = grad_dtype of the call), read-only
 *   m_codes  int8 [numel],  m_scales fp16 bits [ceil(numel/32)]
 *   v_codes  uint8 [numel], v_scales fp16 bits [ceil(numel/32)]
 * All-zero codes and scales are the valid initial state (quantized zeros). */
typedef struct {
  uint16_t* param;
  void* rho;
  const void* grad;
  int8_t* m_codes;
  uint16_t* m_scales;
  uint8_t* v_codes;
  uint16_t* v_scales;
  int64_t numel;
} fo_tensor;

/* "code/flashsim/flash_adamw_sim.py", `FlashAdamWSim.step` (Algorithm 4),
 * for every tensor of the list in one kernel launch and one pass over HBM:
 *   prologue  m = dequant(m), v = dequant(v), theta = reconstruct(theta', rho),
 *             g = fp32(grad);
 *   update    if wd != 0: theta *= (1 - lr wd);
 *             m = b1 m + (1-b1) g;  v = b2 v + ((1-b2) g) g;
 *             theta -= (lr m/(1-b1^t)) / (sqrt(v/(1-b2^t)) + eps);
 *   epilogue  m, v re-quantized with fresh group scales (MOMENTUM / VARIANCE
 *             specs); theta re-split into theta' and rho.
 * Scalars are formed in double on the host and rounded once to fp32.  `step`
 * is t, already incremented (t >= 1 on the first call).  0 <= beta < 1, and
 * lr, eps, weight_decay finite.  `tensors` is a HOST array of n_tensors
 * entries (read during the call only); lists longer than
 * fo_max_tensors_per_launch() are processed in several launches.  Buffers
 * written by the call must not overlap each other or any grad
 * (FO_ERR_ALIAS). */
fo_status fo_adamw_step(const fo_tensor* tensors, int n_tensors, fo_dtype grad_dtype, double lr,
                        double beta1, double beta2, double eps, double weight_decay, int64_t step,
                        int rho_bits, void* stream);

/* ---- the step in the ablation formats ------------------------------------
 * "code/flashsim/flash_adamw_sim.py", `FlashAdamWSim` with its ablation
 * switches: `master_weight_bits` in {24, 32, None}, an fp32 parameter,
 * `companded` and `quantize_states`.  Same update as fo_adamw_step (Algorithm
 * 4, scalars formed in double and rounded once), in any combination of:
 *   parameter  FO_PARAM_BF16_RHO8   bf16 theta' + int8 rho (24-bit master)
 *              FO_PARAM_BF16_RHO16  bf16 theta' + int16 rho (32-bit master)
 *              FO_PARAM_BF16        bf16 parameter, no split (master_weight_bits
 *                                   None): theta = the parameter, written back
 *                                   rounded to nearest even
 *              FO_PARAM_F32         fp32 parameter, no split
 *   states     FO_STATE_COMPANDED   MOMENTUM / VARIANCE specs (as fo_adamw_step)
 *              FO_STATE_LINEAR      MOMENTUM_LINEAR / VARIANCE_LINEAR specs:
 *                                   plain group-32 absmax codes of m and of v
 *              FO_STATE_F32         fp32 m and v, no scales (quantize_states
 *                                   False)
 * Every result is the exact binary32 definition: divisions and square roots
 * correctly rounded from certified approximations, codes, the 24-bit master
 * and a bf16 parameter without a split certified, each with the IEEE chain
 * as fallback (the same bits).  Every format runs in fo_adamw_step's
 * pipelined kernel, which reports a bounded wait that ran out through
 * fo_device_status(); a split master with FO_STATE_COMPANDED gives
 * fo_adamw_step's bits.
 * Buffers as in fo_tensor, with widths by format: param 2 or 4 bytes per
 * element, rho 1 or 2 (unused, may be NULL, without a split), m and v 1 byte
 * (codes) or 4 (fp32), m_scales / v_scales fp16 [ceil(numel/32)] (unused, may
 * be NULL, for fp32 states).  All 16-byte aligned.  Same errors as
 * fo_adamw_step. */
typedef enum {
  FO_PARAM_BF16_RHO8 = 0,
  FO_PARAM_BF16_RHO16 = 1,
  FO_PARAM_BF16 = 2,
  FO_PARAM_F32 = 3
} fo_param_format;
typedef enum { FO_STATE_COMPANDED = 0, FO_STATE_LINEAR = 1, FO_STATE_F32 = 2 } fo_state_format;
typedef struct {
  void* param;
  void* rho;
  const void* grad;
  void* m;
  uint16_t* m_scales;
  void* v;
  uint16_t* v_scales;
  int64_t numel;
} fo_tensor_general;
fo_status fo_adamw_step_general(const fo_tensor_general* tensors, int n_tensors, fo_param_format param_format,
                                fo_state_format state_format, fo_dtype grad_dtype, double lr, double beta1,
                                double beta2, double eps, double weight_decay, int64_t step, void* stream);

/* ---- FlashSGD --------------------------------------------------------------
 * The pages name FlashSGD only in the byte accounting of
 * "code/flashsim/flash_adamw_sim.py" (`bytes_per_param`: theta' + rho and one
 * quantized state, the momentum).  The update read here is SGD with momentum
 * as torch.optim.SGD computes it (dampening 0, no Nesterov, weight decay added
 * to the gradient), every operation rounded once:
 *   g = fp32(grad); if weight_decay != 0: g = g + wd * theta;
 *   buf = momentum * buf + g;  theta = theta - lr * buf
 * lr, momentum, weight_decay are rounded once to fp32.  The buffer lives in
 * fo_tensor_general.m / m_scales in the given state format (FO_STATE_COMPANDED
 * = the MOMENTUM spec, FO_STATE_LINEAR = MOMENTUM_LINEAR, FO_STATE_F32 = fp32);
 * v and v_scales are unused (may be NULL).  All-zero codes and scales are the
 * initial buffer, so the first step stores buf = g as torch does.
 * Every format runs in the pipelined kernel of fo_adamw_step, one HBM pass,
 * momentum codes certified from a hardware reciprocal with the exact chain
 * as fallback (the same bits).  Same errors as fo_adamw_step_general; a
 * bounded wait that ran out is reported through fo_device_status(). */
fo_status fo_sgd_step(const fo_tensor_general* tensors, int n_tensors, fo_param_format param_format,
                      fo_state_format state_format, fo_dtype grad_dtype, double lr, double momentum,
                      double weight_decay, void* stream);

/* Largest tensor list fo_adamw_step handles in a single kernel launch. */
int fo_max_tensors_per_launch(void);

/* Device-side status of fo_adamw_step on the current device, then cleared.
 * The step kernel never waits without a limit: if a bulk load it waits for
 * has not arrived after a bounded number of polls, that block stops and sets
 * bit 0 (FO_DEVICE_WAIT_TIMEOUT); its tiles are then left unprocessed.  The
 * call synchronizes with the device (it copies one word), so use it for
 * diagnostics, not on the hot path.  *status = 0 means no such event. */
#define FO_DEVICE_WAIT_TIMEOUT 1u
fo_status fo_device_status(uint32_t* status);

/* Failure detection without a fault (no counterpart on the pages).  Launches
 * one block that waits, with the step kernel's bounded mbarrier wait, on a
 * barrier that nothing completes; after `polls` unsuccessful polls (1 ..
 * 2^22, the step kernel's own limit) it gives up and sets bit 0 of the device
 * status word, as the step kernel does when one of its waits runs out.  The
 * context stays usable.  FO_ERR_INVALID_ARG for polls out of range; a launch
 * failure gives FO_ERR_CUDA. */
fo_status fo_check_wait_timeout(uint32_t polls, void* stream);

/* ---- allocation-free step -------------------------------------------------
 * No counterpart on the pages: an interface of this library.  Same arguments,
 * results and errors as fo_adamw_step, for a list of at most
 * FO_STATIC_MAX_TENSORS tensors, always in a single launch, and without
 * allocating anything: the tensor list travels in a fixed device array of the
 * library (about 74 KB per device) instead of the kernel's parameter block,
 * and the host side works in fixed static storage.  It serves callers that
 * must not allocate when they step, e.g. a loop that reserves all device
 * memory for its own pools up front, or code that runs while an allocator's
 * lock is held.
 *   - n_tensors > FO_STATIC_MAX_TENSORS returns FO_ERR_TOO_LARGE before any
 *     other check or CUDA call.
 *   - Set-up: the first call on each device looks up the device address of
 *     the array (cudaGetSymbolAddress) and loads every kernel variant this
 *     entry point can launch, with its launch attributes, so that no later
 *     call on that device loads a kernel (with lazy module loading, a
 *     kernel's first use may allocate).  FO_ERR_CUDA if that fails.  Make
 *     the first call on a device before any stream capture.
 *   - Each call copies the list into the array (cudaMemcpyAsync on `stream`,
 *     from pageable host memory, so the host waits until the copy has been
 *     staged) and launches on the same stream.  Nothing in the array has to
 *     start at zero: each call writes every field its launch reads.
 *   - The array and the host staging are shared by all calls: calls that
 *     overlap in time (several host threads, or streams not ordered with one
 *     another) race.  Issue them from one thread on one stream, or order them. */
#define FO_STATIC_MAX_TENSORS 1024
fo_status fo_adamw_step_static(const fo_tensor* tensors, int n_tensors, fo_dtype grad_dtype, double lr,
                               double beta1, double beta2, double eps, double weight_decay, int64_t step,
                               int rho_bits, void* stream);

#ifdef __cplusplus
}
#endif
#endif
