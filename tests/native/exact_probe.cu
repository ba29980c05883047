// exact_probe.cu -- test helper: the correctly rounded division and square
// root of the step kernel (fo_device.cuh: div_const, sqrt_cert, div_cert)
// against the device's IEEE operations (__fdiv_rn, __fsqrt_rn), bit for bit,
// over every input of their stated domains (sqrt, constant divisors) or a
// dense structured sweep (general division).  A result whose certificate
// failed is not compared (the step recomputes it); the number of failed
// certificates is reported.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "fo_device.cuh"

using fo::ConstDivisor;

struct Counts {
  unsigned long long checked, mismatched, uncertain;
};

__device__ __forceinline__ void tally(Counts* c, unsigned long long checked, unsigned long long bad,
                                      unsigned long long unsure) {
  for (int o = 16; o > 0; o >>= 1) {
    checked += __shfl_xor_sync(0xffffffffu, checked, o);
    bad += __shfl_xor_sync(0xffffffffu, bad, o);
    unsure += __shfl_xor_sync(0xffffffffu, unsure, o);
  }
  if ((threadIdx.x & 31) == 0) {
    atomicAdd(&c->checked, checked);
    atomicAdd(&c->mismatched, bad);
    atomicAdd(&c->uncertain, unsure);
  }
}

// every positive pattern (and +0) in {+0} U [2^-95, 2^100]
__global__ void sqrt_kernel(Counts* out) {
  const uint32_t lo = 0x10000000u;  // 2^-95
  const uint32_t hi = 0x71800000u;  // 2^100
  unsigned long long n = 0, bad = 0, unsure = 0;
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t b = (uint64_t)lo - 1 + blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; b <= hi; b += stride) {
    const float x = b == (uint64_t)lo - 1 ? 0.0f : __uint_as_float((uint32_t)b);
    bool ok = true;
    const float s = fo::sqrt_cert(x, ok);
    ++n;
    if (!ok) ++unsure;
    else if (__float_as_uint(s) != __float_as_uint(__fsqrt_rn(x))) ++bad;
  }
  tally(out, n, bad, unsure);
}

// every pattern with a = +0 or 2^-80 <= |a| <= 2^100, one divisor per launch
__global__ void div_const_kernel(ConstDivisor c, float b, Counts* out) {
  const uint32_t lo = 0x17800000u;  // 2^-80
  const uint32_t hi = 0x71800000u;  // 2^100
  const uint64_t span = (uint64_t)(hi - lo) + 1;
  unsigned long long n = 0, bad = 0;
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < 2 * span + 1; i += stride) {
    float a;
    if (i == 2 * span) a = 0.0f;
    else a = __uint_as_float((uint32_t)(lo + (i % span)) | (i >= span ? 0x80000000u : 0u));
    const float q = fo::div_const(a, c);
    ++n;
    if (__float_as_uint(q) != __float_as_uint(__fdiv_rn(a, b))) ++bad;
  }
  tally(out, n, bad, 0);
}

// General division n / d: for each divisor d of the list, every numerator
// significand of one binade, with an exponent that keeps the quotient in
// range, both signs, and n = +0.
__global__ void div_cert_kernel(const float* divisors, int nd, Counts* out) {
  unsigned long long n = 0, bad = 0, unsure = 0;
  const uint64_t per = (uint64_t)1 << 24;  // 2^23 significands x 2 signs
  const uint64_t total = per * (uint64_t)nd;
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < total; i += stride) {
    const int k = (int)(i / per);
    const uint32_t r = (uint32_t)(i % per);
    const float d = divisors[k];
    // numerator exponent: spread over [-80, 69] by the divisor index, then
    // clipped so that |n/d| >= 2^-101
    int e = -80 + (int)((k * 37) % 150);
    const int ed = (int)((__float_as_uint(d) >> 23) & 0xFF) - 127;
    if (e - ed < -100) e = ed - 100;
    const uint32_t bits = ((uint32_t)(e + 127) << 23) | (r & 0x7FFFFFu) | ((r >> 23) << 31);
    const float num = (r == 0 && (k & 1)) ? 0.0f : __uint_as_float(bits);
    bool ok = true;
    const float q = fo::div_cert(num, d, ok);
    ++n;
    if (!ok) ++unsure;
    else if (__float_as_uint(q) != __float_as_uint(__fdiv_rn(num, d))) ++bad;
  }
  tally(out, n, bad, unsure);
}

static int run(void (*launch)(Counts*), unsigned long long* host) {
  Counts* d = nullptr;
  if (cudaMalloc(&d, sizeof(Counts)) != cudaSuccess) return 1;
  cudaMemset(d, 0, sizeof(Counts));
  launch(d);
  cudaError_t e = cudaDeviceSynchronize();
  Counts c{};
  if (e == cudaSuccess) e = cudaMemcpy(&c, d, sizeof(Counts), cudaMemcpyDeviceToHost);
  cudaFree(d);
  host[0] = c.checked;
  host[1] = c.mismatched;
  host[2] = c.uncertain;
  return e == cudaSuccess ? 0 : 2;
}

extern "C" int probe_sqrt(unsigned long long* host) {
  return run([](Counts* d) { sqrt_kernel<<<152 * 8, 256>>>(d); }, host);
}

// host[3 * i ..] for divisor i
extern "C" int probe_div_const(const float* divisors, int nd, unsigned long long* host) {
  for (int i = 0; i < nd; ++i) {
    const float b = divisors[i];
    const ConstDivisor c = fo::const_divisor(b);
    Counts* d = nullptr;
    if (cudaMalloc(&d, sizeof(Counts)) != cudaSuccess) return 1;
    cudaMemset(d, 0, sizeof(Counts));
    div_const_kernel<<<152 * 8, 256>>>(c, b, d);
    cudaError_t e = cudaDeviceSynchronize();
    Counts h{};
    if (e == cudaSuccess) e = cudaMemcpy(&h, d, sizeof(Counts), cudaMemcpyDeviceToHost);
    cudaFree(d);
    if (e != cudaSuccess) return 2;
    host[3 * i] = h.checked;
    host[3 * i + 1] = h.mismatched;
    host[3 * i + 2] = h.uncertain;
  }
  return 0;
}

extern "C" int probe_div_cert(const float* divisors, int nd, unsigned long long* host) {
  float* dd = nullptr;
  if (cudaMalloc(&dd, nd * sizeof(float)) != cudaSuccess) return 1;
  cudaMemcpy(dd, divisors, nd * sizeof(float), cudaMemcpyHostToDevice);
  Counts* d = nullptr;
  if (cudaMalloc(&d, sizeof(Counts)) != cudaSuccess) return 1;
  cudaMemset(d, 0, sizeof(Counts));
  div_cert_kernel<<<152 * 8, 256>>>(dd, nd, d);
  cudaError_t e = cudaDeviceSynchronize();
  Counts h{};
  if (e == cudaSuccess) e = cudaMemcpy(&h, d, sizeof(Counts), cudaMemcpyDeviceToHost);
  cudaFree(d);
  cudaFree(dd);
  host[0] = h.checked;
  host[1] = h.mismatched;
  host[2] = h.uncertain;
  return e == cudaSuccess ? 0 : 2;
}
