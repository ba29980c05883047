// fo_host.h -- host-side helpers shared by the entry points of libfo.so.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "fo.h"
#include "fo_device.cuh"

namespace fo {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int64_t n_groups(int64_t n) { return (n + 31) / 32; }

// Remember the CUDA error of the calling thread's last failed launch.
void record_cuda_error(cudaError_t e);

// Turn the state after a launch into a status (FO_ERR_CUDA on a launch error).
inline fo_status launch_status() {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return FO_ERR_CUDA;
  }
  return FO_OK;
}

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// Python-float scalars of the AdamW update, each formed in double and rounded
// once to fp32 (as torch does for scalar operands of fp32 tensor arithmetic).
struct StepScalars {
  float c_wd, b1, one_minus_b1, b2, one_minus_b2, bc1, bc2, lr, eps;
  // constants of the approximate update: RN(lr * RN(1/bc1)) and RN(sqrt(RN(1/bc2)))
  float lr_ib1, sqrt_ib2;
  // the exact update of the fused kernel: division by bc1 and bc2, and the
  // gradient gate G (a gradient with 0 < |g| < G sends its thread to the
  // exact IEEE chain)
  ConstDivisor d1, d2;
  float gate;
  float c255_root_bc2;  // RN(255 sqrt(bc2)): companded variance codes from the exact sqrt(v_hat)
  float neg_zero;  // -0.0f: the addend of an exact product (RN(a b) = fma(a, b, -0))
  // 1 when lr, eps, the betas and the bias corrections lie in the ranges the
  // exact update is proved for; 0 sends every element to the IEEE chain
  int fast;
};
StepScalars step_scalars(double lr, double beta1, double beta2, double eps, double weight_decay, int64_t step);

// State formats of a pipelined launch: companded codes, linear codes, or
// fp32 states without scales.
constexpr int kStatesCompanded = 0, kStatesLinear = 1, kStatesF32 = 2;

// SGD with momentum through the pipelined step kernel, for the parameter
// format rho_bits (8 or 16: a split master; 0: a bf16 parameter; 32: an fp32
// parameter) and the state format `states`; the list must already have
// passed the checks of fo_sgd_step.
fo_status launch_sgd_fast(const fo_tensor_general* tensors, int n_tensors, bool grad_bf16, int rho_bits, int states,
                          double lr, double momentum, double weight_decay, cudaStream_t s);

// AdamW through the pipelined step kernel, for the parameter and state
// formats as above; the list must already have passed the checks of
// fo_adamw_step_general.
fo_status launch_adamw_fused(const fo_tensor_general* tensors, int n_tensors, bool grad_bf16, int rho_bits,
                             int states, double lr, double beta1, double beta2, double eps, double weight_decay,
                             int64_t step, cudaStream_t s);

}  // namespace fo
