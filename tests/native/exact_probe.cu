// exact_probe.cu -- test helper: the correctly rounded division and square
// root of the step kernel (fo_device.cuh: div_const2, sqrt_cert2, div_cert2,
// in the packed f32x2 form the kernel runs) against the device's IEEE
// operations (__fdiv_rn, __fsqrt_rn), bit for bit, over every input of their
// stated domains (sqrt, constant divisors) or a dense structured sweep
// (general division).  Each thread evaluates two inputs, one per lane.  A
// result whose certificate failed is not compared (the step recomputes it);
// the number of failed certificates is reported.
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

// every positive pattern (and +0) in {+0} U [2^-95, 2^100]; lane y takes the
// input half the domain above lane x's
__global__ void sqrt_kernel(Counts* out) {
  const uint64_t lo = 0x10000000u;  // 2^-95
  const uint64_t hi = 0x71800000u;  // 2^100
  const uint64_t span = hi - lo + 2;  // +0 and the patterns lo..hi
  const uint64_t half = (span + 1) / 2;
  unsigned long long n = 0, bad = 0, unsure = 0;
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  auto input = [&](uint64_t i) { return i == 0 ? 0.0f : __uint_as_float((uint32_t)(lo + i - 1)); };
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < half; i += stride) {
    const bool two = i + half < span;
    const float2 x = make_float2(input(i), two ? input(i + half) : 1.0f);
    uint32_t bx = 0, by = 0;
    const float2 s = fo::sqrt_cert2<true>(x, bx);
    // the lanes' certificates, told apart by running each lane's input alone too
    fo::sqrt_cert2<true>(make_float2(x.x, x.x), bx);
    fo::sqrt_cert2<true>(make_float2(x.y, x.y), by);
    const bool ok[2] = {(bx >> 31) == 0, (by >> 31) == 0};
    const float got[2] = {s.x, s.y};
    const float in[2] = {x.x, x.y};
    for (int l = 0; l < (two ? 2 : 1); ++l) {
      ++n;
      if (!ok[l]) ++unsure;
      else if (__float_as_uint(got[l]) != __float_as_uint(__fsqrt_rn(in[l]))) ++bad;
    }
  }
  tally(out, n, bad, unsure);
}

// every pattern with a = +0 or 2^-80 <= |a| <= 2^100, one divisor per launch;
// lane y takes the negated dividend of lane x (+0 for a = +0: -0 is outside
// the domain)
__global__ void div_const_kernel(ConstDivisor c, float b, Counts* out) {
  const uint32_t lo = 0x17800000u;  // 2^-80
  const uint32_t hi = 0x71800000u;  // 2^100
  const uint64_t span = (uint64_t)(hi - lo) + 1;
  unsigned long long n = 0, bad = 0;
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < span + 1; i += stride) {
    const float a = i == span ? 0.0f : __uint_as_float((uint32_t)(lo + i));
    const float na = i == span ? 0.0f : -a;
    const float2 q = fo::div_const2<true>(make_float2(a, na), c);
    n += 2;
    if (__float_as_uint(q.x) != __float_as_uint(__fdiv_rn(a, b))) ++bad;
    if (__float_as_uint(q.y) != __float_as_uint(__fdiv_rn(na, b))) ++bad;
  }
  tally(out, n, bad, 0);
}

// General division n / d: for each divisor d of the list, every numerator
// significand of one binade, with an exponent that keeps the quotient in
// range, both signs, and n = +0.  Lane y divides the same numerator by the
// divisor half the list further on.
__device__ __forceinline__ float div_numerator(const float* divisors, int k, uint32_t r) {
  const float d = divisors[k];
  // numerator exponent: spread over [-80, 69] by the divisor index, then
  // clipped so that |n/d| >= 2^-101
  int e = -80 + (int)((k * 37) % 150);
  const int ed = (int)((__float_as_uint(d) >> 23) & 0xFF) - 127;
  if (e - ed < -100) e = ed - 100;
  const uint32_t bits = ((uint32_t)(e + 127) << 23) | (r & 0x7FFFFFu) | ((r >> 23) << 31);
  return (r == 0 && (k & 1)) ? 0.0f : __uint_as_float(bits);
}
__global__ void div_cert_kernel(const float* divisors, int nd, Counts* out) {
  unsigned long long n = 0, bad = 0, unsure = 0;
  const uint64_t per = (uint64_t)1 << 24;  // 2^23 significands x 2 signs
  const int halfd = (nd + 1) / 2;
  const uint64_t total = per * (uint64_t)halfd;
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < total; i += stride) {
    const int k0 = (int)(i / per);
    const int k1 = k0 + halfd;
    const bool two = k1 < nd;
    const uint32_t r = (uint32_t)(i % per);
    const float n0 = div_numerator(divisors, k0, r), d0 = divisors[k0];
    const float n1 = two ? div_numerator(divisors, k1, r) : 1.0f, d1 = two ? divisors[k1] : 1.0f;
    uint32_t b = 0, bx = 0, by = 0;
    const float2 q = fo::div_cert2<true>(make_float2(n0, n1), make_float2(d0, d1), b);
    fo::div_cert2<true>(make_float2(n0, n0), make_float2(d0, d0), bx);
    fo::div_cert2<true>(make_float2(n1, n1), make_float2(d1, d1), by);
    ++n;
    if (bx >> 31) ++unsure;
    else if (__float_as_uint(q.x) != __float_as_uint(__fdiv_rn(n0, d0))) ++bad;
    if (two) {
      ++n;
      if (by >> 31) ++unsure;
      else if (__float_as_uint(q.y) != __float_as_uint(__fdiv_rn(n1, d1))) ++bad;
    }
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
