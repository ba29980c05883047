// fo_step_general.cu -- the FlashAdamW step in every parameter and state
// format of the page "code/flashsim/flash_adamw_sim.py" (`FlashAdamWSim` with
// `master_weight_bits` in {24, 32, None}, an fp32 parameter, `companded` and
// `quantize_states`): the ablations the paper compares the method against.
//
// Every result is the exact IEEE chain of the definition (no approximation,
// so no certification either).  The paper's own format runs in the fast
// kernel of fo_step.cu; this one serves the ablation formats.  One launch
// covers a list of tensors; a block takes a tile of 4096 elements, a thread
// 16 consecutive elements (half a group of 32: the group maximum is one
// shuffle with the neighbouring thread).
#include <cuda_bf16.h>
#include <math.h>

#include <algorithm>
#include <vector>

#include "fo.h"
#include "fo_device.cuh"
#include "fo_host.h"

namespace fo {
namespace {

constexpr int kGenMaxTensors = 400;
constexpr int kGenTile = kThreads * kPerThread;

struct GenArgs {
  StepScalars k;
  int sgd;         // 0: AdamW (Algorithm 4); 1: SGD with momentum (fo_sgd_step)
  float sgd_mu;    // SGD: momentum, and weight decay added to the gradient
  float sgd_wd;
  int param_format;
  int state_format;
  int grad_bf16;
  int decay;
  int n_tensors;
  int64_t total_tiles;
  int64_t tile_start[kGenMaxTensors + 1];
  fo_tensor_general t[kGenMaxTensors];
};
static_assert(sizeof(GenArgs) <= 32764, "kernel parameter block too large");

// RN( RN(lr * RN(m / bc1)) / RN( RN(sqrt(RN(v / bc2))) + eps ) )
__device__ __forceinline__ float general_delta(float m, float v, const StepScalars& k) {
  const float mhat = __fdiv_rn(m, k.bc1);
  const float vhat = __fdiv_rn(v, k.bc2);
  return __fdiv_rn(__fmul_rn(k.lr, mhat), __fadd_rn(__fsqrt_rn(vhat), k.eps));
}

__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

// fp32 -> bf16 bits, round to nearest even (torch's .to(bfloat16)); NaN stays a NaN
__device__ __forceinline__ uint16_t f32_to_bf16_rne(float x) { return __bfloat16_as_ushort(__float2bfloat16_rn(x)); }

__global__ void __launch_bounds__(kThreads) general_step_kernel(const __grid_constant__ GenArgs a) {
  const StepScalars& k = a.k;
  for (int64_t tile = blockIdx.x; tile < a.total_tiles; tile += gridDim.x) {
    int lo = 0, hi = a.n_tensors - 1;  // the tensor owning the tile: last start <= tile
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (a.tile_start[mid] <= tile) lo = mid;
      else hi = mid - 1;
    }
    const fo_tensor_general& T = a.t[lo];
    const int64_t n = T.numel;
    const int64_t e0 = (tile - a.tile_start[lo]) * kGenTile + static_cast<int64_t>(threadIdx.x) * kPerThread;

    float theta[kPerThread], m[kPerThread], v[kPerThread];
#pragma unroll
    for (int j = 0; j < kPerThread; ++j) {
      theta[j] = 0.0f;
      m[j] = 0.0f;
      v[j] = 0.0f;
      const int64_t i = e0 + j;
      if (i >= n) continue;  // the zero padding of a ragged last group
      const float g = a.grad_bf16 ? bf16_to_f32(static_cast<const uint16_t*>(T.grad)[i])
                                  : static_cast<const float*>(T.grad)[i];
      // prologue: theta, m, v
      switch (a.param_format) {
        case FO_PARAM_BF16_RHO8:
          theta[j] = reconstruct_one<8>(static_cast<const uint16_t*>(T.param)[i],
                                        static_cast<int>(static_cast<const int8_t*>(T.rho)[i]));
          break;
        case FO_PARAM_BF16_RHO16:
          theta[j] = reconstruct_one<16>(static_cast<const uint16_t*>(T.param)[i],
                                         static_cast<int>(static_cast<const int16_t*>(T.rho)[i]));
          break;
        case FO_PARAM_BF16: theta[j] = bf16_to_f32(static_cast<const uint16_t*>(T.param)[i]); break;
        default: theta[j] = static_cast<const float*>(T.param)[i]; break;
      }
      float mj, vj;
      if (a.sgd) {
        // SGD with momentum: the buffer is the m state; v is not used
        if (a.state_format == FO_STATE_F32) {
          mj = static_cast<const float*>(T.m)[i];
        } else {
          const int qm = static_cast<int>(static_cast<const int8_t*>(T.m)[i]);
          const float sm = f16_bits_to_f32(T.m_scales[i / kGroup]);
          mj = __fmul_rn(a.state_format == FO_STATE_COMPANDED ? code_unit_value<true, true>(qm)
                                                              : code_unit_value<true, false>(qm),
                         sm);
        }
        const float gd = a.decay ? __fadd_rn(g, __fmul_rn(a.sgd_wd, theta[j])) : g;
        mj = __fadd_rn(__fmul_rn(a.sgd_mu, mj), gd);
        theta[j] = __fsub_rn(theta[j], __fmul_rn(k.lr, mj));
        m[j] = mj;
        continue;
      }
      if (a.state_format == FO_STATE_F32) {
        mj = static_cast<const float*>(T.m)[i];
        vj = static_cast<const float*>(T.v)[i];
      } else {
        const int qm = static_cast<int>(static_cast<const int8_t*>(T.m)[i]);
        const int qv = static_cast<int>(static_cast<const uint8_t*>(T.v)[i]);
        const float sm = f16_bits_to_f32(T.m_scales[i / kGroup]);
        const float sv = f16_bits_to_f32(T.v_scales[i / kGroup]);
        if (a.state_format == FO_STATE_COMPANDED) {
          mj = __fmul_rn(code_unit_value<true, true>(qm), sm);
          const float u = __fmul_rn(code_unit_value<false, false>(qv), sv);
          vj = __fmul_rn(u, u);
        } else {
          mj = __fmul_rn(code_unit_value<true, false>(qm), sm);
          vj = __fmul_rn(code_unit_value<false, false>(qv), sv);
        }
      }
      // the update, each operation rounded once
      if (a.decay) theta[j] = __fmul_rn(theta[j], k.c_wd);
      mj = __fadd_rn(__fmul_rn(k.b1, mj), __fmul_rn(k.one_minus_b1, g));
      vj = __fadd_rn(__fmul_rn(k.b2, vj), __fmul_rn(__fmul_rn(k.one_minus_b2, g), g));
      theta[j] = __fsub_rn(theta[j], general_delta(mj, vj, k));
      m[j] = mj;
      v[j] = vj;
    }

    // epilogue: states
    if (a.state_format == FO_STATE_F32) {
#pragma unroll
      for (int j = 0; j < kPerThread; ++j) {
        if (e0 + j >= n) continue;
        static_cast<float*>(T.m)[e0 + j] = m[j];
        if (!a.sgd) static_cast<float*>(T.v)[e0 + j] = v[j];
      }
    } else {
      const bool companded = a.state_format == FO_STATE_COMPANDED;
      float r[kPerThread];  // what the variance codes encode: sqrt(v) or v
#pragma unroll
      for (int j = 0; j < kPerThread; ++j) r[j] = companded ? __fsqrt_rn(v[j]) : v[j];
      float am = fabsf(m[0]), av = r[0];
#pragma unroll
      for (int j = 1; j < kPerThread; ++j) {
        am = keep_first_max(am, fabsf(m[j]));
        av = keep_first_max(av, r[j]);
      }
      am = group_max_pair(am);
      av = group_max_pair(av);
      const uint16_t sm16 = f32_to_f16_bits(am);
      const uint16_t sv16 = f32_to_f16_bits(av);
      const float dm = guarded_divisor(sm16), dv = guarded_divisor(sv16);
#pragma unroll
      for (int j = 0; j < kPerThread; ++j) {
        if (e0 + j >= n) continue;
        static_cast<int8_t*>(T.m)[e0 + j] = static_cast<int8_t>(
            companded ? encode_code<true, true>(m[j], dm) : encode_code<true, false>(m[j], dm));
        if (!a.sgd) static_cast<uint8_t*>(T.v)[e0 + j] = static_cast<uint8_t>(encode_code<false, false>(r[j], dv));
      }
      if (e0 < n && !(threadIdx.x & 1)) {
        T.m_scales[e0 / kGroup] = sm16;
        if (!a.sgd) T.v_scales[e0 / kGroup] = sv16;
      }
    }

    // epilogue: the parameter
#pragma unroll
    for (int j = 0; j < kPerThread; ++j) {
      const int64_t i = e0 + j;
      if (i >= n) continue;
      switch (a.param_format) {
        case FO_PARAM_BF16_RHO8: {
          uint16_t h;
          int rho;
          split_one<8>(theta[j], h, rho);
          static_cast<uint16_t*>(T.param)[i] = h;
          static_cast<int8_t*>(T.rho)[i] = static_cast<int8_t>(rho);
          break;
        }
        case FO_PARAM_BF16_RHO16: {
          uint16_t h;
          int rho;
          split_one<16>(theta[j], h, rho);
          static_cast<uint16_t*>(T.param)[i] = h;
          static_cast<int16_t*>(T.rho)[i] = static_cast<int16_t>(rho);
          break;
        }
        case FO_PARAM_BF16: static_cast<uint16_t*>(T.param)[i] = f32_to_bf16_rne(theta[j]); break;
        default: static_cast<float*>(T.param)[i] = theta[j]; break;
      }
    }
  }
}

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

}  // namespace
}  // namespace fo

using namespace fo;

namespace fo {
namespace {

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

// Launches over the list, 400 tensors per launch; `args` carries the scalars
// and formats.
fo_status launch_general(const fo_tensor_general* tensors, int n_tensors, GenArgs& args, cudaStream_t s) {
  int sms = 152, dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int i = 0;
  while (i < n_tensors) {
    int cnt = 0;
    int64_t tiles = 0;
    for (; i < n_tensors && cnt < kGenMaxTensors; ++i) {
      if (tensors[i].numel == 0) continue;
      args.tile_start[cnt] = tiles;
      args.t[cnt] = tensors[i];
      tiles += (tensors[i].numel + kGenTile - 1) / kGenTile;
      ++cnt;
    }
    if (cnt == 0) break;
    args.tile_start[cnt] = tiles;
    args.n_tensors = cnt;
    args.total_tiles = tiles;
    const unsigned grid = static_cast<unsigned>(std::min<int64_t>(tiles, static_cast<int64_t>(sms) * 8));
    general_step_kernel<<<grid, kThreads, 0, s>>>(args);
    const fo_status st = launch_status();
    if (st != FO_OK) return st;
  }
  return FO_OK;
}

}  // namespace
}  // namespace fo

extern "C" fo_status fo_adamw_step_general(const fo_tensor_general* tensors, int n_tensors, fo_param_format param_format,
                                           fo_state_format state_format, fo_dtype grad_dtype, double lr, double beta1,
                                           double beta2, double eps, double weight_decay, int64_t step, void* stream) {
  fo_status st = check_general(tensors, n_tensors, param_format, state_format, grad_dtype, true);
  if (st != FO_OK) return st;
  if (step < 1) return FO_ERR_INVALID_ARG;
  if (!std::isfinite(lr) || !std::isfinite(eps) || !std::isfinite(weight_decay)) return FO_ERR_INVALID_ARG;
  if (!(beta1 >= 0.0 && beta1 < 1.0) || !(beta2 >= 0.0 && beta2 < 1.0)) return FO_ERR_INVALID_ARG;
  GenArgs args;
  args.k = step_scalars(lr, beta1, beta2, eps, weight_decay, step);
  args.sgd = 0;
  args.sgd_mu = args.sgd_wd = 0.0f;
  args.param_format = param_format;
  args.state_format = state_format;
  args.grad_bf16 = grad_dtype == FO_DT_BF16;
  args.decay = weight_decay != 0.0;
  return launch_general(tensors, n_tensors, args, as_stream(stream));
}

extern "C" fo_status fo_sgd_step(const fo_tensor_general* tensors, int n_tensors, fo_param_format param_format,
                                 fo_state_format state_format, fo_dtype grad_dtype, double lr, double momentum,
                                 double weight_decay, void* stream) {
  fo_status st = check_general(tensors, n_tensors, param_format, state_format, grad_dtype, false);
  if (st != FO_OK) return st;
  if (!std::isfinite(lr) || !std::isfinite(momentum) || !std::isfinite(weight_decay)) return FO_ERR_INVALID_ARG;
  if (state_format == FO_STATE_COMPANDED &&
      (param_format == FO_PARAM_BF16_RHO8 || param_format == FO_PARAM_BF16_RHO16))
    return launch_sgd_fast(tensors, n_tensors, grad_dtype == FO_DT_BF16, param_format == FO_PARAM_BF16_RHO8 ? 8 : 16,
                           lr, momentum, weight_decay, as_stream(stream));
  GenArgs args;
  args.k = step_scalars(lr, 0.0, 0.0, 1.0, 0.0, 1);  // only k.lr is used: RN(lr)
  args.sgd = 1;
  args.sgd_mu = static_cast<float>(momentum);
  args.sgd_wd = static_cast<float>(weight_decay);
  args.param_format = param_format;
  args.state_format = state_format;
  args.grad_bf16 = grad_dtype == FO_DT_BF16;
  args.decay = weight_decay != 0.0;
  return launch_general(tensors, n_tensors, args, as_stream(stream));
}
