// fo_step_general.cu -- the FlashAdamW step in every parameter and state
// format of the page "code/flashsim/flash_adamw_sim.py" (`FlashAdamWSim` with
// `master_weight_bits` in {24, 32, None}, an fp32 parameter, `companded` and
// `quantize_states`): the ablations the paper compares the method against.
//
// Every result equals the exact IEEE chain of the definition.  Codes, the
// 24-bit master and a bf16 parameter without a split come from certified
// approximations with an in-thread exact fallback, as in the fused kernel;
// everything else is computed exactly.  The
// paper's own format runs in the fused kernel of fo_step.cu; this one serves
// the ablation formats.  One launch covers a list of tensors, with one kernel
// instantiation per format; a block takes a tile of 4096 elements, a thread
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
  int fast_theta;  // AdamW with the 24-bit master or a bf16 parameter, eps >= 2^-40: certified theta
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

// Certification constants, as in the fused kernel (fo_step.cu): a new theta
// from the approximate update is accepted when both ends of the interval
// theta - (delta' +- E), E = 2^-19 |delta'| + 2^-100, round to the same 24-bit
// master; a code when its approximate argument is more than 2^-10 away from
// every half-integer.  Uncertain results are recomputed in-thread through the
// exact chain.
constexpr float kGenDeltaRel = 0x1p-19f;
constexpr float kGenDeltaAbs = 0x1p-100f;

// Rare exact fallbacks kept out of line, so that the unrolled element loop
// stays small enough for the instruction cache (measured: the bf16-parameter
// and code formats gain 3-12 %; the 24-bit master's fallback stays inline,
// where a call made the fp32-state format 9 % slower).
__device__ __noinline__ float exact_theta(float theta, float m, float v, StepScalars k) {
  return __fsub_rn(theta, general_delta(m, v, k));
}
template <bool kSigned, bool kSoftsign>
__device__ __noinline__ uint32_t exact_code(float r, float divisor) {
  return static_cast<uint8_t>(encode_code<kSigned, kSoftsign>(r, divisor));
}

// Inputs of one element as values: gradient, master weight, old m and v.
struct GenIn {
  float g, theta, m, v;
};

// The inputs of element i with scalar loads (ragged chunks).
template <int PF, int SF, bool SGD, bool GB>
__device__ __forceinline__ GenIn load_one(const fo_tensor_general& T, int64_t i, const float* lut_m, const float* lut_v) {
  constexpr bool kQuant = SF != FO_STATE_F32;
  GenIn r;
  r.g = GB ? bf16_to_f32(static_cast<const uint16_t*>(T.grad)[i]) : static_cast<const float*>(T.grad)[i];
  if (PF == FO_PARAM_BF16_RHO8)
    r.theta = reconstruct_one<8>(static_cast<const uint16_t*>(T.param)[i],
                                 static_cast<int>(static_cast<const int8_t*>(T.rho)[i]));
  else if (PF == FO_PARAM_BF16_RHO16)
    r.theta = reconstruct_one<16>(static_cast<const uint16_t*>(T.param)[i],
                                  static_cast<int>(static_cast<const int16_t*>(T.rho)[i]));
  else if (PF == FO_PARAM_BF16) r.theta = bf16_to_f32(static_cast<const uint16_t*>(T.param)[i]);
  else r.theta = static_cast<const float*>(T.param)[i];
  r.v = 0.0f;
  if (kQuant) {
    r.m = __fmul_rn(lut_m[static_cast<const uint8_t*>(T.m)[i]], f16_bits_to_f32(T.m_scales[i / kGroup]));
    if (!SGD) r.v = __fmul_rn(lut_v[static_cast<const uint8_t*>(T.v)[i]], f16_bits_to_f32(T.v_scales[i / kGroup]));
  } else {
    r.m = static_cast<const float*>(T.m)[i];
    if (!SGD) r.v = static_cast<const float*>(T.v)[i];
  }
  return r;
}

// 4 * Q consecutive words from 16-byte-aligned global memory.
template <int Q>
__device__ __forceinline__ void ld_words(const void* p, uint32_t* w) {
#pragma unroll
  for (int q = 0; q < Q; ++q) {
    const uint4 x = reinterpret_cast<const uint4*>(p)[q];
    w[4 * q] = x.x; w[4 * q + 1] = x.y; w[4 * q + 2] = x.z; w[4 * q + 3] = x.w;
  }
}
template <int Q>
__device__ __forceinline__ void st_words(void* p, const uint32_t* w) {
#pragma unroll
  for (int q = 0; q < Q; ++q)
    reinterpret_cast<uint4*>(p)[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
}

// One kernel per (parameter format, state format, optimizer, gradient type).
// A thread takes 16 consecutive elements (half a group of 32): 128-bit loads
// and stores for a whole chunk, scalar ones for a tensor's ragged end.
// Resident blocks per SM each instantiation is compiled for: four (at most
// 64 registers, spilling a few hundred bytes to L1) where the parameter is a
// plain bf16 or fp32 value, two (at most 128) where the master is split,
// whose longer chains lose more to spills than they gain from occupancy.
template <int PF>
constexpr int kGenMinBlocks = (PF == FO_PARAM_BF16 || PF == FO_PARAM_F32) ? 4 : 2;

template <int PF, int SF, bool SGD, bool GB>
__global__ void __launch_bounds__(kThreads, kGenMinBlocks<PF>) general_step_kernel(const __grid_constant__ GenArgs a) {
  constexpr bool kQuant = SF != FO_STATE_F32;
  constexpr bool kComp = SF == FO_STATE_COMPANDED;
  constexpr int kP = kPerThread;
  const StepScalars& k = a.k;
  // unit value of every code byte, with the element-wise definition's operations
  __shared__ float lut_m[256], lut_v[256];
  static_assert(kThreads == 256, "one table entry per thread");
  if (kQuant) {
    const int q = static_cast<int>(threadIdx.x);
    const int qs = static_cast<int>(static_cast<int8_t>(q));
    lut_m[q] = kComp ? code_unit_value<true, true>(qs) : code_unit_value<true, false>(qs);
    lut_v[q] = code_unit_value<false, false>(q);
  }
  __syncthreads();
  for (int64_t tile = blockIdx.x; tile < a.total_tiles; tile += gridDim.x) {
    int lo = 0, hi = a.n_tensors - 1;  // the tensor owning the tile: last start <= tile
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (a.tile_start[mid] <= tile) lo = mid;
      else hi = mid - 1;
    }
    const fo_tensor_general& T = a.t[lo];
    const int64_t n = T.numel;
    const int64_t e0 = (tile - a.tile_start[lo]) * kGenTile + static_cast<int64_t>(threadIdx.x) * kP;
    const bool full = e0 + kP <= n;

    // ------------------------------------------------------------ inputs
    uint32_t gw[GB ? 8 : 16], pw[PF == FO_PARAM_F32 ? 16 : 8], rw[PF == FO_PARAM_BF16_RHO16 ? 8 : 4];
    uint32_t mw[kQuant ? 4 : 16], vw[kQuant ? 4 : 16];
    float s_m = 0.0f, s_v = 0.0f;
    if (full) {
      ld_words<GB ? 2 : 4>(static_cast<const char*>(T.grad) + e0 * (GB ? 2 : 4), gw);
      ld_words<PF == FO_PARAM_F32 ? 4 : 2>(static_cast<const char*>(T.param) + e0 * (PF == FO_PARAM_F32 ? 4 : 2), pw);
      if (PF == FO_PARAM_BF16_RHO8) ld_words<1>(static_cast<const char*>(T.rho) + e0, rw);
      if (PF == FO_PARAM_BF16_RHO16) ld_words<2>(static_cast<const char*>(T.rho) + e0 * 2, rw);
      ld_words<kQuant ? 1 : 4>(static_cast<const char*>(T.m) + e0 * (kQuant ? 1 : 4), mw);
      if (!SGD) ld_words<kQuant ? 1 : 4>(static_cast<const char*>(T.v) + e0 * (kQuant ? 1 : 4), vw);
      if (kQuant) {
        s_m = f16_bits_to_f32(T.m_scales[e0 / kGroup]);
        if (!SGD) s_v = f16_bits_to_f32(T.v_scales[e0 / kGroup]);
      }
    }

    // ------------------------------------------------------------ update
    float theta[kP], m[kP], v[kP];
    uint32_t w24[kP];  // split word of the new theta (24-bit master)
#pragma unroll
    for (int j = 0; j < kP; ++j) {
      theta[j] = 0.0f;
      m[j] = 0.0f;
      v[j] = 0.0f;
      w24[j] = 0u;
      GenIn in;
      if (full) {
        const uint32_t gb = GB ? ((gw[j >> 1] >> (16 * (j & 1))) & 0xFFFFu) : 0u;
        in.g = GB ? bf16_to_f32(static_cast<uint16_t>(gb)) : __uint_as_float(gw[j]);
        if (PF == FO_PARAM_F32) {
          in.theta = __uint_as_float(pw[j]);
        } else {
          const uint16_t ph = static_cast<uint16_t>((pw[j >> 1] >> (16 * (j & 1))) & 0xFFFFu);
          if (PF == FO_PARAM_BF16_RHO8)
            in.theta = reconstruct_one<8>(ph, static_cast<int>(static_cast<int8_t>((rw[j >> 2] >> (8 * (j & 3))) & 0xFFu)));
          else if (PF == FO_PARAM_BF16_RHO16)
            in.theta = reconstruct_one<16>(ph, static_cast<int>(static_cast<int16_t>((rw[j >> 1] >> (16 * (j & 1))) & 0xFFFFu)));
          else
            in.theta = bf16_to_f32(ph);
        }
        in.v = 0.0f;
        if (kQuant) {
          in.m = __fmul_rn(lut_m[(mw[j >> 2] >> (8 * (j & 3))) & 0xFFu], s_m);
          if (!SGD) in.v = __fmul_rn(lut_v[(vw[j >> 2] >> (8 * (j & 3))) & 0xFFu], s_v);
        } else {
          in.m = __uint_as_float(mw[j]);
          if (!SGD) in.v = __uint_as_float(vw[j]);
        }
      } else {
        if (e0 + j >= n) continue;  // the zero padding of a ragged last group
        in = load_one<PF, SF, SGD, GB>(T, e0 + j, lut_m, lut_v);
      }
      if (kComp && !SGD) in.v = __fmul_rn(in.v, in.v);  // the variance codes hold sqrt(v)
      float th = in.theta, mj = in.m;
      if (SGD) {
        // SGD with momentum: the buffer is the m state; v is not used
        const float gd = a.decay ? __fadd_rn(in.g, __fmul_rn(a.sgd_wd, th)) : in.g;
        mj = __fadd_rn(__fmul_rn(a.sgd_mu, mj), gd);
        th = __fsub_rn(th, __fmul_rn(k.lr, mj));
        if (PF == FO_PARAM_BF16_RHO8) w24[j] = split_word<8>(th);
      } else {
        // the update, each operation rounded once
        if (a.decay) th = __fmul_rn(th, k.c_wd);
        mj = __fadd_rn(__fmul_rn(k.b1, mj), __fmul_rn(k.one_minus_b1, in.g));
        const float vj = __fadd_rn(__fmul_rn(k.b2, in.v), __fmul_rn(__fmul_rn(k.one_minus_b2, in.g), in.g));
        if (PF == FO_PARAM_BF16_RHO8 && a.fast_theta) {
          const float den = __fadd_rn(__fmul_rn(sqrt_approx(vj), k.sqrt_ib2), k.eps);
          const float dl = __fmul_rn(__fmul_rn(mj, k.lr_ib1), rcp_approx(den));
          const float e = __fmaf_rn(fabsf(dl), kGenDeltaRel, kGenDeltaAbs);
          const uint32_t wl = __float_as_uint(__fsub_rn(th, __fadd_rn(dl, e))) + 0x8080u;
          const uint32_t wh = __float_as_uint(__fsub_rn(th, __fsub_rn(dl, e))) + 0x8080u;
          w24[j] = (wl ^ wh) > 0xFFu ? split_word<8>(__fsub_rn(th, general_delta(mj, vj, k))) : wl;
        } else if (PF == FO_PARAM_BF16 && a.fast_theta) {
          // bf16 parameter: the same interval, rounded to nearest even bf16
          // (monotone too); one bf16 for both ends is the exact result's
          const float den = __fadd_rn(__fmul_rn(sqrt_approx(vj), k.sqrt_ib2), k.eps);
          const float dl = __fmul_rn(__fmul_rn(mj, k.lr_ib1), rcp_approx(den));
          const float e = __fmaf_rn(fabsf(dl), kGenDeltaRel, kGenDeltaAbs);
          const uint16_t bl = f32_to_bf16_rne(__fsub_rn(th, __fadd_rn(dl, e)));
          const uint16_t bh = f32_to_bf16_rne(__fsub_rn(th, __fsub_rn(dl, e)));
          th = bl == bh ? __uint_as_float(static_cast<uint32_t>(bl) << 16) : exact_theta(th, mj, vj, k);
        } else {
          th = __fsub_rn(th, general_delta(mj, vj, k));
          if (PF == FO_PARAM_BF16_RHO8) w24[j] = split_word<8>(th);
        }
        v[j] = vj;
      }
      theta[j] = th;
      m[j] = mj;
    }

    // ------------------------------------------------------------ states
    if (!kQuant) {
      if (full) {
        uint32_t o[16];
#pragma unroll
        for (int j = 0; j < kP; ++j) o[j] = __float_as_uint(m[j]);
        st_words<4>(static_cast<float*>(T.m) + e0, o);
        if (!SGD) {
#pragma unroll
          for (int j = 0; j < kP; ++j) o[j] = __float_as_uint(v[j]);
          st_words<4>(static_cast<float*>(T.v) + e0, o);
        }
      } else {
#pragma unroll
        for (int j = 0; j < kP; ++j) {
          if (e0 + j >= n) continue;
          static_cast<float*>(T.m)[e0 + j] = m[j];
          if (!SGD) static_cast<float*>(T.v)[e0 + j] = v[j];
        }
      }
    } else {
      // group maxima; with companding the variance codes encode sqrt(v), and
      // RN(sqrt(max v)) is the maximum of RN(sqrt(v)) (monotone square root)
      float am = fabsf(m[0]), av = v[0];
#pragma unroll
      for (int j = 1; j < kP; ++j) {
        am = keep_first_max(am, fabsf(m[j]));
        av = keep_first_max(av, v[j]);
      }
      am = group_max_pair(am);
      av = group_max_pair(av);
      if (kComp) av = __fsqrt_rn(av);
      const uint16_t sm16 = f32_to_f16_bits(am);
      const uint16_t sv16 = f32_to_f16_bits(av);
      const float dm = guarded_divisor(sm16), dv = guarded_divisor(sv16);
      // certified codes (group constants, at most one hardware approximation
      // per argument), exact where an argument is close to a half-integer
      const float rs = __fdiv_rn(1.0f, dm);
      const float c1 = __fmul_rn(254.0f, rs);
      const float c127 = __fdiv_rn(127.0f, dm);
      const float c2 = __fdiv_rn(255.0f, dv);
      uint32_t cmw[4] = {0u, 0u, 0u, 0u}, cvw[4] = {0u, 0u, 0u, 0u};
#pragma unroll
      for (int j = 0; j < kP; ++j) {
        bool near;
        const float tm = kComp ? momentum_t_approx(m[j], rs, c1) : fminf(fmaxf(__fmul_rn(m[j], c127), -127.0f), 127.0f);
        uint32_t cm = round_code_certified(tm, near);
        if (near) cm = kComp ? exact_code<true, true>(m[j], dm) : exact_code<true, false>(m[j], dm);
        cmw[j >> 2] |= cm << (8 * (j & 3));
        if (!SGD) {
          const float tv = variance_t_approx_from_root(kComp ? sqrt_approx(v[j]) : v[j], c2);
          uint32_t cv = round_code_certified(tv, near);
          if (near) cv = exact_code<false, false>(kComp ? __fsqrt_rn(v[j]) : v[j], dv);
          cvw[j >> 2] |= cv << (8 * (j & 3));
        }
      }
      if (full) {
        st_words<1>(static_cast<uint8_t*>(T.m) + e0, cmw);
        if (!SGD) st_words<1>(static_cast<uint8_t*>(T.v) + e0, cvw);
      } else {
#pragma unroll
        for (int j = 0; j < kP; ++j) {
          if (e0 + j >= n) continue;
          static_cast<uint8_t*>(T.m)[e0 + j] = static_cast<uint8_t>(cmw[j >> 2] >> (8 * (j & 3)));
          if (!SGD) static_cast<uint8_t*>(T.v)[e0 + j] = static_cast<uint8_t>(cvw[j >> 2] >> (8 * (j & 3)));
        }
      }
      if (e0 < n && !(threadIdx.x & 1)) {
        T.m_scales[e0 / kGroup] = sm16;
        if (!SGD) T.v_scales[e0 / kGroup] = sv16;
      }
    }

    // ------------------------------------------------------------ parameter
    uint32_t po[PF == FO_PARAM_F32 ? 16 : 8], ro[PF == FO_PARAM_BF16_RHO16 ? 8 : 4];
#pragma unroll
    for (int q = 0; q < (PF == FO_PARAM_BF16_RHO16 ? 8 : 4); ++q) ro[q] = 0u;
#pragma unroll
    for (int j = 0; j < kP; ++j) {
      uint32_t hbits = 0u;
      if (PF == FO_PARAM_BF16_RHO8) {
        hbits = w24[j] >> 16;
        ro[j >> 2] |= (((w24[j] >> 8) ^ 0x80u) & 0xFFu) << (8 * (j & 3));
      } else if (PF == FO_PARAM_BF16_RHO16) {
        uint16_t h;
        int rho;
        split_one<16>(theta[j], h, rho);
        hbits = h;
        ro[j >> 1] |= (static_cast<uint32_t>(rho) & 0xFFFFu) << (16 * (j & 1));
      } else if (PF == FO_PARAM_BF16) {
        hbits = f32_to_bf16_rne(theta[j]);
      }
      if (PF == FO_PARAM_F32) po[j] = __float_as_uint(theta[j]);
      else if (j & 1) po[j >> 1] |= hbits << 16;
      else po[j >> 1] = hbits;
    }
    if (full) {
      st_words<PF == FO_PARAM_F32 ? 4 : 2>(static_cast<char*>(T.param) + e0 * (PF == FO_PARAM_F32 ? 4 : 2), po);
      if (PF == FO_PARAM_BF16_RHO8) st_words<1>(static_cast<char*>(T.rho) + e0, ro);
      if (PF == FO_PARAM_BF16_RHO16) st_words<2>(static_cast<char*>(T.rho) + e0 * 2, ro);
    } else {
#pragma unroll
      for (int j = 0; j < kP; ++j) {
        const int64_t i = e0 + j;
        if (i >= n) continue;
        if (PF == FO_PARAM_F32) {
          static_cast<float*>(T.param)[i] = theta[j];
        } else {
          static_cast<uint16_t*>(T.param)[i] = static_cast<uint16_t>(po[j >> 1] >> (16 * (j & 1)));
          if (PF == FO_PARAM_BF16_RHO8) static_cast<uint8_t*>(T.rho)[i] = static_cast<uint8_t>(ro[j >> 2] >> (8 * (j & 3)));
          if (PF == FO_PARAM_BF16_RHO16)
            static_cast<uint16_t*>(T.rho)[i] = static_cast<uint16_t>(ro[j >> 1] >> (16 * (j & 1)));
        }
      }
    }
  }
}

// The instantiation for a format, by table lookup.
using GenKernel = void (*)(GenArgs);
template <int PF, int SF, bool SGD>
constexpr GenKernel gen_kernel(bool gb) {
  return gb ? general_step_kernel<PF, SF, SGD, true> : general_step_kernel<PF, SF, SGD, false>;
}
template <int PF, bool SGD>
GenKernel gen_kernel_sf(int sf, bool gb) {
  return sf == FO_STATE_COMPANDED ? gen_kernel<PF, FO_STATE_COMPANDED, SGD>(gb)
         : sf == FO_STATE_LINEAR  ? gen_kernel<PF, FO_STATE_LINEAR, SGD>(gb)
                                  : gen_kernel<PF, FO_STATE_F32, SGD>(gb);
}
// Formats with codes run in the pipelined kernel (fo_step.cu); here only the
// fp32-state forms.
template <bool SGD>
GenKernel gen_kernel_pf(int pf, int sf, bool gb) {
  (void)sf;
  return pf == FO_PARAM_BF16_RHO8    ? gen_kernel<FO_PARAM_BF16_RHO8, FO_STATE_F32, SGD>(gb)
         : pf == FO_PARAM_BF16_RHO16 ? gen_kernel<FO_PARAM_BF16_RHO16, FO_STATE_F32, SGD>(gb)
         : pf == FO_PARAM_BF16       ? gen_kernel<FO_PARAM_BF16, FO_STATE_F32, SGD>(gb)
                                     : gen_kernel<FO_PARAM_F32, FO_STATE_F32, SGD>(gb);
}

// The pipelined kernel's parameter format (its kRhoBits) of a format.
int fused_param_format(int pf) {
  return pf == FO_PARAM_BF16_RHO8 ? 8 : pf == FO_PARAM_BF16_RHO16 ? 16 : pf == FO_PARAM_BF16 ? 0 : 32;
}
GenKernel select_general_kernel(const GenArgs& a) {
  return a.sgd ? gen_kernel_pf<true>(a.param_format, a.state_format, a.grad_bf16)
               : gen_kernel_pf<false>(a.param_format, a.state_format, a.grad_bf16);
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
    select_general_kernel(args)<<<grid, kThreads, 0, s>>>(args);
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
  // every format with codes: the pipelined kernel
  if (state_format != FO_STATE_F32)
    return launch_adamw_fused(tensors, n_tensors, grad_dtype == FO_DT_BF16, fused_param_format(param_format),
                              state_format == FO_STATE_COMPANDED, lr, beta1, beta2, eps, weight_decay, step,
                              as_stream(stream));
  GenArgs args;
  args.k = step_scalars(lr, beta1, beta2, eps, weight_decay, step);
  args.sgd = 0;
  args.sgd_mu = args.sgd_wd = 0.0f;
  args.param_format = param_format;
  args.state_format = state_format;
  args.grad_bf16 = grad_dtype == FO_DT_BF16;
  args.decay = weight_decay != 0.0;
  args.fast_theta = (param_format == FO_PARAM_BF16_RHO8 || param_format == FO_PARAM_BF16) && args.k.eps >= 0x1p-40f;
  return launch_general(tensors, n_tensors, args, as_stream(stream));
}

extern "C" fo_status fo_sgd_step(const fo_tensor_general* tensors, int n_tensors, fo_param_format param_format,
                                 fo_state_format state_format, fo_dtype grad_dtype, double lr, double momentum,
                                 double weight_decay, void* stream) {
  fo_status st = check_general(tensors, n_tensors, param_format, state_format, grad_dtype, false);
  if (st != FO_OK) return st;
  if (!std::isfinite(lr) || !std::isfinite(momentum) || !std::isfinite(weight_decay)) return FO_ERR_INVALID_ARG;
  if (state_format != FO_STATE_F32)
    return launch_sgd_fast(tensors, n_tensors, grad_dtype == FO_DT_BF16, fused_param_format(param_format),
                           state_format == FO_STATE_COMPANDED, lr, momentum, weight_decay, as_stream(stream));
  GenArgs args;
  args.k = step_scalars(lr, 0.0, 0.0, 1.0, 0.0, 1);  // only k.lr is used: RN(lr)
  args.sgd = 1;
  args.fast_theta = 0;
  args.sgd_mu = static_cast<float>(momentum);
  args.sgd_wd = static_cast<float>(weight_decay);
  args.param_format = param_format;
  args.state_format = state_format;
  args.grad_bf16 = grad_dtype == FO_DT_BF16;
  args.decay = weight_decay != 0.0;
  return launch_general(tensors, n_tensors, args, as_stream(stream));
}
