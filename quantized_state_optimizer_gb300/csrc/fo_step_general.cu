// fo_step_general.cu -- the FlashAdamW and FlashSGD steps in every parameter
// and state format of the page "code/flashsim/flash_adamw_sim.py"
// (`FlashAdamWSim` with `master_weight_bits` in {24, 32, None}, an fp32
// parameter, `companded` and `quantize_states`): the ablations the paper
// compares the method against.  The argument checks of the two entry points;
// every format runs in the pipelined step kernel of fo_step.cu, instantiated
// per parameter format (split master with int8 or int16 rho, bf16, fp32) and
// state format (companded codes, linear codes, fp32 states).
#include <math.h>

#include <algorithm>
#include <cmath>
#include <vector>

#include "fo.h"
#include "fo_device.cuh"
#include "fo_host.h"

namespace fo {
namespace {

int param_bytes(int f) { return f == FO_PARAM_F32 ? 4 : 2; }
int rho_bytes(int f) { return f == FO_PARAM_BF16_RHO8 ? 1 : f == FO_PARAM_BF16_RHO16 ? 2 : 0; }
int state_bytes(int f) { return f == FO_STATE_F32 ? 4 : 1; }

// Writable buffers must not overlap anything; grads may overlap each other.
bool general_overlap(const fo_tensor_general* ts, int n, int pf, int sf, int grad_bytes, bool with_v) {
  struct Range {
    uintptr_t lo, hi;
    bool writable;
  };
  std::vector<Range> r;
  r.reserve(static_cast<size_t>(n) * 7);
  for (int i = 0; i < n; ++i) {
    const fo_tensor_general& t = ts[i];
    if (t.numel == 0) continue;
    const uintptr_t e = static_cast<uintptr_t>(t.numel);
    const uintptr_t g = static_cast<uintptr_t>(n_groups(t.numel));
    auto add = [&](const void* p, uintptr_t bytes, bool w) {
      const uintptr_t b = reinterpret_cast<uintptr_t>(p);
      r.push_back({b, b + bytes, w});
    };
    add(t.param, param_bytes(pf) * e, true);
    if (rho_bytes(pf)) add(t.rho, rho_bytes(pf) * e, true);
    add(t.grad, grad_bytes * e, false);
    add(t.m, state_bytes(sf) * e, true);
    if (with_v) add(t.v, state_bytes(sf) * e, true);
    if (sf != FO_STATE_F32) {
      add(t.m_scales, 2 * g, true);
      if (with_v) add(t.v_scales, 2 * g, true);
    }
  }
  std::sort(r.begin(), r.end(), [](const Range& x, const Range& y) { return x.lo < y.lo; });
  uintptr_t max_any = 0, max_w = 0;
  for (const Range& x : r) {
    if (x.lo < max_w) return true;
    if (x.writable && x.lo < max_any) return true;
    max_any = std::max(max_any, x.hi);
    if (x.writable) max_w = std::max(max_w, x.hi);
  }
  return false;
}


// Checks shared by both entry points; `with_v` is false for SGD (one state).
fo_status check_general(const fo_tensor_general* tensors, int n_tensors, int param_format, int state_format,
                        int grad_dtype, bool with_v) {
  if (n_tensors < 0 || (n_tensors > 0 && !tensors)) return FO_ERR_INVALID_ARG;
  if (param_format < FO_PARAM_BF16_RHO8 || param_format > FO_PARAM_F32) return FO_ERR_INVALID_ARG;
  if (state_format < FO_STATE_COMPANDED || state_format > FO_STATE_F32) return FO_ERR_INVALID_ARG;
  if (grad_dtype != FO_DT_F32 && grad_dtype != FO_DT_BF16) return FO_ERR_INVALID_ARG;
  const bool quantized = state_format != FO_STATE_F32;
  const bool has_rho = param_format == FO_PARAM_BF16_RHO8 || param_format == FO_PARAM_BF16_RHO16;
  for (int i = 0; i < n_tensors; ++i) {
    const fo_tensor_general& t = tensors[i];
    if (t.numel < 0) return FO_ERR_INVALID_ARG;
    if (t.numel == 0) continue;
    if (!t.param || !t.grad || !t.m || (with_v && !t.v) || (has_rho && !t.rho) ||
        (quantized && (!t.m_scales || (with_v && !t.v_scales))))
      return FO_ERR_INVALID_ARG;
    if (!aligned16(t.param) || !aligned16(t.grad) || !aligned16(t.m) || (with_v && !aligned16(t.v)) ||
        (has_rho && !aligned16(t.rho)) ||
        (quantized && (!aligned16(t.m_scales) || (with_v && !aligned16(t.v_scales)))))
      return FO_ERR_MISALIGNED;
  }
  if (general_overlap(tensors, n_tensors, param_format, state_format, grad_dtype == FO_DT_BF16 ? 2 : 4, with_v))
    return FO_ERR_ALIAS;
  return FO_OK;
}

// The pipelined kernel's parameter format (its kRhoBits) and state format.
int fused_param_format(int pf) {
  return pf == FO_PARAM_BF16_RHO8 ? 8 : pf == FO_PARAM_BF16_RHO16 ? 16 : pf == FO_PARAM_BF16 ? 0 : 32;
}
int fused_state_format(int sf) {
  return sf == FO_STATE_COMPANDED ? kStatesCompanded : sf == FO_STATE_LINEAR ? kStatesLinear : kStatesF32;
}

}  // namespace
}  // namespace fo

using namespace fo;

extern "C" fo_status fo_adamw_step_general(const fo_tensor_general* tensors, int n_tensors, fo_param_format param_format,
                                           fo_state_format state_format, fo_dtype grad_dtype, double lr, double beta1,
                                           double beta2, double eps, double weight_decay, int64_t step, void* stream) {
  fo_status st = check_general(tensors, n_tensors, param_format, state_format, grad_dtype, true);
  if (st != FO_OK) return st;
  if (step < 1) return FO_ERR_INVALID_ARG;
  if (!std::isfinite(lr) || !std::isfinite(eps) || !std::isfinite(weight_decay)) return FO_ERR_INVALID_ARG;
  if (!(beta1 >= 0.0 && beta1 < 1.0) || !(beta2 >= 0.0 && beta2 < 1.0)) return FO_ERR_INVALID_ARG;
  return launch_adamw_fused(tensors, n_tensors, grad_dtype == FO_DT_BF16, fused_param_format(param_format),
                            fused_state_format(state_format), lr, beta1, beta2, eps, weight_decay, step,
                            as_stream(stream));
}

extern "C" fo_status fo_sgd_step(const fo_tensor_general* tensors, int n_tensors, fo_param_format param_format,
                                 fo_state_format state_format, fo_dtype grad_dtype, double lr, double momentum,
                                 double weight_decay, void* stream) {
  fo_status st = check_general(tensors, n_tensors, param_format, state_format, grad_dtype, false);
  if (st != FO_OK) return st;
  if (!std::isfinite(lr) || !std::isfinite(momentum) || !std::isfinite(weight_decay)) return FO_ERR_INVALID_ARG;
  return launch_sgd_fast(tensors, n_tensors, grad_dtype == FO_DT_BF16, fused_param_format(param_format),
                         fused_state_format(state_format), lr, momentum, weight_decay, as_stream(stream));
}
