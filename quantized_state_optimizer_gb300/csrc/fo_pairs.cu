// fo_pairs.cu -- the two standalone kernel pairs of libfo.so:
//   fo_quantize / fo_dequantize   ("code/flashsim/quantization.py",
//                                  `quantize` and `dequantize`, Alg. 2-3)
//   fo_split / fo_reconstruct     ("code/gpu/equivalence.py", `eq_ecc`:
//                                  compute_ecc_bits / reconstruct_fp32_param)
// All four are elementwise streams over HBM: one thread per 16 elements,
// 128-bit loads and stores, a group of 32 shared by two neighbouring lanes.
#include <string>

#include <algorithm>

#include "fo.h"
#include "fo_device.cuh"
#include "fo_host.h"

namespace fo {

namespace {
thread_local std::string g_last_cuda_error;
}

void record_cuda_error(cudaError_t e) {
  g_last_cuda_error = std::string(cudaGetErrorName(e)) + ": " + cudaGetErrorString(e);
}

// ------------------------------------------------------------- quantize
template <bool kSigned, bool kSqrt, bool kSoftsign>
__global__ void __launch_bounds__(kThreads)
    quantize_kernel(const float* __restrict__ x, int64_t n, void* __restrict__ codes,
                    uint16_t* __restrict__ scales) {
  const int64_t e0 = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) * kPerThread;
  float r[kPerThread];
  if (e0 + kPerThread <= n) {
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      V16B w;
      w.q = ld_stream(x + e0 + 4 * v);
#pragma unroll
      for (int k = 0; k < 4; ++k) r[4 * v + k] = w.f32[k];
    }
  } else {
    // ragged end: elements past n are the zero padding of the last group
#pragma unroll
    for (int j = 0; j < kPerThread; ++j) r[j] = (e0 + j < n) ? x[e0 + j] : 0.0f;
  }
  // Group maximum of |x| (signed specs) or x.  With the square root, the
  // group's value is RN(sqrt(max x)): a correctly rounded square root is
  // monotone, so that is the maximum of RN(sqrt(x)) over the group.
  float a = kSigned ? fabsf(r[0]) : r[0];
#pragma unroll
  for (int j = 1; j < kPerThread; ++j) a = keep_first_max(a, kSigned ? fabsf(r[j]) : r[j]);
  a = group_max_pair(a);
  if (kSqrt) a = __fsqrt_rn(a);
  const uint16_t s16 = f32_to_f16_bits(a);
  const float safe = guarded_divisor(s16);

  // Certified approximate codes, exact where uncertain.  The code argument t
  // (127 softsign(x/s), 127 x/s, 255 sqrt(x)/s or 255 x/s) comes from group
  // constants and at most one hardware approximation; its error is far below
  // the margin that round_code_certified leaves around every half-integer.
  V16B out;
  {
    const float rs = __fdiv_rn(1.0f, safe);
    const float c1 = __fmul_rn(254.0f, rs);
    const float c2 = __fdiv_rn(255.0f, safe);
    const float c127 = __fdiv_rn(127.0f, safe);
    uint32_t near = 0;
#pragma unroll
    for (int j = 0; j < kPerThread; ++j) {
      bool nj;
      float t;
      if (kSigned && kSoftsign) t = momentum_t_approx(r[j], rs, c1);
      else if (kSigned) t = fminf(fmaxf(__fmul_rn(r[j], c127), -127.0f), 127.0f);
      else t = variance_t_approx_from_root(kSqrt ? sqrt_approx(r[j]) : r[j], c2);
      out.u8[j] = round_code_certified(t, nj);
      if (nj) near |= 1u << j;
    }
    if (near) {
#pragma unroll
      for (int j = 0; j < kPerThread; ++j)
        if (near & (1u << j))
          out.u8[j] = static_cast<uint8_t>(encode_code<kSigned, kSoftsign>(kSqrt ? __fsqrt_rn(r[j]) : r[j], safe));
    }
  }
  uint8_t* c = static_cast<uint8_t*>(codes);
  if (e0 + kPerThread <= n) {
    st_stream(c + e0, out.q);
  } else {
#pragma unroll
    for (int j = 0; j < kPerThread; ++j)
      if (e0 + j < n) c[e0 + j] = out.u8[j];
  }
  if (!(threadIdx.x & 1) && e0 < n) scales[e0 / kGroup] = s16;
}

// ----------------------------------------------------------- dequantize
template <bool kSigned, bool kSqrt, bool kSoftsign>
__global__ void __launch_bounds__(kThreads)
    dequantize_kernel(const void* __restrict__ codes, const uint16_t* __restrict__ scales,
                      int64_t n, float* __restrict__ out) {
  // unit value of every code byte, with the element-wise definition's operations
  __shared__ float lut[256];
  static_assert(kThreads == 256, "one table entry per thread");
  lut[threadIdx.x] = code_unit_value<kSigned, kSoftsign>(kSigned ? static_cast<int>(static_cast<int8_t>(threadIdx.x))
                                                                 : static_cast<int>(threadIdx.x));
  __syncthreads();
  // grid-stride over chunks of kThreads * kPerThread elements (the table is
  // built once per block)
  const uint8_t* c = static_cast<const uint8_t*>(codes);
  for (int64_t e0 = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) * kPerThread; e0 < n;
       e0 += static_cast<int64_t>(gridDim.x) * kThreads * kPerThread) {
    V16B w;
    const bool full = e0 + kPerThread <= n;
    if (full) {
      w.q = ld_stream(c + e0);
    } else {
#pragma unroll
      for (int j = 0; j < kPerThread; ++j) w.u8[j] = (e0 + j < n) ? c[e0 + j] : 0;
    }
    const float s = f16_bits_to_f32(scales[e0 / kGroup]);
    float o[kPerThread];
#pragma unroll
    for (int j = 0; j < kPerThread; ++j) {
      float y = __fmul_rn(lut[w.u8[j]], s);
      if (kSqrt) y = __fmul_rn(y, y);
      o[j] = y;
    }
    if (full) {
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        V16B t;
#pragma unroll
        for (int k = 0; k < 4; ++k) t.f32[k] = o[4 * v + k];
        st_stream(out + e0 + 4 * v, t.q);
      }
    } else {
#pragma unroll
      for (int j = 0; j < kPerThread; ++j)
        if (e0 + j < n) out[e0 + j] = o[j];
    }
  }
}

// ---------------------------------------------------------------- split
template <int kRhoBits>
__global__ void __launch_bounds__(kThreads)
    split_kernel(const float* __restrict__ theta, int64_t n, uint16_t* __restrict__ hi_out,
                 void* __restrict__ rho_out) {
  const int64_t e0 = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) * kPerThread;
  if (e0 >= n) return;
  const bool full = e0 + kPerThread <= n;
  float x[kPerThread];
  if (full) {
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      V16B w;
      w.q = ld_stream(theta + e0 + 4 * v);
#pragma unroll
      for (int k = 0; k < 4; ++k) x[4 * v + k] = w.f32[k];
    }
  } else {
#pragma unroll
    for (int j = 0; j < kPerThread; ++j) x[j] = (e0 + j < n) ? theta[e0 + j] : 0.0f;
  }
  V16B h[2], r[2];
#pragma unroll
  for (int j = 0; j < kPerThread; ++j) {
    uint16_t hi;
    int rho;
    split_one<kRhoBits>(x[j], hi, rho);
    h[j / 8].u16[j % 8] = hi;
    if (kRhoBits == 8) r[0].i8[j] = static_cast<int8_t>(rho);
    else r[j / 8].i16[j % 8] = static_cast<int16_t>(rho);
  }
  if (full) {
    st_stream(hi_out + e0, h[0].q);
    st_stream(hi_out + e0 + 8, h[1].q);
    if (kRhoBits == 8) {
      st_stream(static_cast<int8_t*>(rho_out) + e0, r[0].q);
    } else {
      st_stream(static_cast<int16_t*>(rho_out) + e0, r[0].q);
      st_stream(static_cast<int16_t*>(rho_out) + e0 + 8, r[1].q);
    }
  } else {
#pragma unroll
    for (int j = 0; j < kPerThread; ++j) {
      if (e0 + j >= n) continue;
      hi_out[e0 + j] = h[j / 8].u16[j % 8];
      if (kRhoBits == 8) static_cast<int8_t*>(rho_out)[e0 + j] = r[0].i8[j];
      else static_cast<int16_t*>(rho_out)[e0 + j] = r[j / 8].i16[j % 8];
    }
  }
}

// ---------------------------------------------------------- reconstruct
template <int kRhoBits>
__global__ void __launch_bounds__(kThreads)
    reconstruct_kernel(const uint16_t* __restrict__ hi_in, const void* __restrict__ rho_in,
                       int64_t n, float* __restrict__ theta) {
  const int64_t e0 = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) * kPerThread;
  if (e0 >= n) return;
  const bool full = e0 + kPerThread <= n;
  V16B h[2], r[2];
  if (full) {
    h[0].q = ld_stream(hi_in + e0);
    h[1].q = ld_stream(hi_in + e0 + 8);
    if (kRhoBits == 8) {
      r[0].q = ld_stream(static_cast<const int8_t*>(rho_in) + e0);
    } else {
      r[0].q = ld_stream(static_cast<const int16_t*>(rho_in) + e0);
      r[1].q = ld_stream(static_cast<const int16_t*>(rho_in) + e0 + 8);
    }
  } else {
#pragma unroll
    for (int j = 0; j < kPerThread; ++j) {
      const bool live = e0 + j < n;
      h[j / 8].u16[j % 8] = live ? hi_in[e0 + j] : 0;
      if (kRhoBits == 8) r[0].i8[j] = live ? static_cast<const int8_t*>(rho_in)[e0 + j] : 0;
      else r[j / 8].i16[j % 8] = live ? static_cast<const int16_t*>(rho_in)[e0 + j] : 0;
    }
  }
  float o[kPerThread];
#pragma unroll
  for (int j = 0; j < kPerThread; ++j) {
    const int rho = kRhoBits == 8 ? static_cast<int>(r[0].i8[j]) : static_cast<int>(r[j / 8].i16[j % 8]);
    o[j] = reconstruct_one<kRhoBits>(h[j / 8].u16[j % 8], rho);
  }
  if (full) {
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      V16B t;
#pragma unroll
      for (int k = 0; k < 4; ++k) t.f32[k] = o[4 * v + k];
      st_stream(theta + e0 + 4 * v, t.q);
    }
  } else {
#pragma unroll
    for (int j = 0; j < kPerThread; ++j)
      if (e0 + j < n) theta[e0 + j] = o[j];
  }
}

inline unsigned blocks_for(int64_t n) {
  return static_cast<unsigned>((n + kTile - 1) / kTile);
}

}  // namespace fo

using namespace fo;

extern "C" {

const char* fo_status_string(fo_status s) {
  switch (s) {
    case FO_OK: return "FO_OK";
    case FO_ERR_INVALID_ARG: return "FO_ERR_INVALID_ARG";
    case FO_ERR_MISALIGNED: return "FO_ERR_MISALIGNED";
    case FO_ERR_CUDA: return "FO_ERR_CUDA";
    case FO_ERR_ALIAS: return "FO_ERR_ALIAS";
    case FO_ERR_TOO_LARGE: return "FO_ERR_TOO_LARGE";
  }
  return "FO_ERR_UNKNOWN";
}

const char* fo_last_cuda_error(void) { return g_last_cuda_error.c_str(); }

fo_status fo_quantize(const float* x, int64_t n, fo_spec spec, void* codes, uint16_t* scales,
                      void* stream) {
  if (n < 0 || spec < FO_SPEC_MOMENTUM || spec > FO_SPEC_VARIANCE_LINEAR) return FO_ERR_INVALID_ARG;
  if (n == 0) return FO_OK;
  if (!x || !codes || !scales) return FO_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(codes) || !aligned16(scales)) return FO_ERR_MISALIGNED;
  const unsigned grid = blocks_for(n);
  cudaStream_t s = as_stream(stream);
  switch (spec) {
    case FO_SPEC_MOMENTUM: quantize_kernel<true, false, true><<<grid, kThreads, 0, s>>>(x, n, codes, scales); break;
    case FO_SPEC_VARIANCE: quantize_kernel<false, true, false><<<grid, kThreads, 0, s>>>(x, n, codes, scales); break;
    case FO_SPEC_MOMENTUM_LINEAR: quantize_kernel<true, false, false><<<grid, kThreads, 0, s>>>(x, n, codes, scales); break;
    case FO_SPEC_VARIANCE_LINEAR: quantize_kernel<false, false, false><<<grid, kThreads, 0, s>>>(x, n, codes, scales); break;
  }
  return launch_status();
}

fo_status fo_dequantize(const void* codes, const uint16_t* scales, int64_t n, fo_spec spec,
                        float* out, void* stream) {
  if (n < 0 || spec < FO_SPEC_MOMENTUM || spec > FO_SPEC_VARIANCE_LINEAR) return FO_ERR_INVALID_ARG;
  if (n == 0) return FO_OK;
  if (!codes || !scales || !out) return FO_ERR_INVALID_ARG;
  if (!aligned16(codes) || !aligned16(scales) || !aligned16(out)) return FO_ERR_MISALIGNED;
  int sms = 152, dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const unsigned grid = std::min<unsigned>(blocks_for(n), static_cast<unsigned>(sms) * 8);  // 8 blocks per SM
  cudaStream_t s = as_stream(stream);
  switch (spec) {
    case FO_SPEC_MOMENTUM: dequantize_kernel<true, false, true><<<grid, kThreads, 0, s>>>(codes, scales, n, out); break;
    case FO_SPEC_VARIANCE: dequantize_kernel<false, true, false><<<grid, kThreads, 0, s>>>(codes, scales, n, out); break;
    case FO_SPEC_MOMENTUM_LINEAR: dequantize_kernel<true, false, false><<<grid, kThreads, 0, s>>>(codes, scales, n, out); break;
    case FO_SPEC_VARIANCE_LINEAR: dequantize_kernel<false, false, false><<<grid, kThreads, 0, s>>>(codes, scales, n, out); break;
  }
  return launch_status();
}

fo_status fo_split(const float* theta, int64_t n, int rho_bits, uint16_t* theta_bf16, void* rho,
                   void* stream) {
  if (n < 0 || (rho_bits != 8 && rho_bits != 16)) return FO_ERR_INVALID_ARG;
  if (n == 0) return FO_OK;
  if (!theta || !theta_bf16 || !rho) return FO_ERR_INVALID_ARG;
  if (!aligned16(theta) || !aligned16(theta_bf16) || !aligned16(rho)) return FO_ERR_MISALIGNED;
  const unsigned grid = blocks_for(n);
  cudaStream_t s = as_stream(stream);
  if (rho_bits == 8) split_kernel<8><<<grid, kThreads, 0, s>>>(theta, n, theta_bf16, rho);
  else split_kernel<16><<<grid, kThreads, 0, s>>>(theta, n, theta_bf16, rho);
  return launch_status();
}

fo_status fo_reconstruct(const uint16_t* theta_bf16, const void* rho, int64_t n, int rho_bits,
                         float* theta, void* stream) {
  if (n < 0 || (rho_bits != 8 && rho_bits != 16)) return FO_ERR_INVALID_ARG;
  if (n == 0) return FO_OK;
  if (!theta || !theta_bf16 || !rho) return FO_ERR_INVALID_ARG;
  if (!aligned16(theta) || !aligned16(theta_bf16) || !aligned16(rho)) return FO_ERR_MISALIGNED;
  const unsigned grid = blocks_for(n);
  cudaStream_t s = as_stream(stream);
  if (rho_bits == 8) reconstruct_kernel<8><<<grid, kThreads, 0, s>>>(theta_bf16, rho, n, theta);
  else reconstruct_kernel<16><<<grid, kThreads, 0, s>>>(theta_bf16, rho, n, theta);
  return launch_status();
}

}  // extern "C"
