// approx_probe.cu -- test helper: worst-case error, in units in the last
// place, of the hardware approximations the step kernel certifies
// (rcp.approx.ftz.f32, sqrt.approx.ftz.f32, rsqrt.approx.ftz.f32) against the
// correctly rounded IEEE results, over every positive normal fp32 input.
#include <cuda_runtime.h>
#include <stdint.h>

__device__ __forceinline__ float rcp_apx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ float sqrt_apx(float x) {
  float r;
  asm("sqrt.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ float rsqrt_apx(float x) {
  float r;
  asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// inputs: bits in [0x00800000, 0x7F800000) (all positive normals); one thread
// per input, grid-stride.  out[0] = max ulp error of rcp, out[1] = of sqrt,
// out[2] = max relative error of rsqrt, |y sqrt(x) - 1|, in units of 2^-24
// (rounded up): with y^2 = hi + lo exactly (hi = RN(y y), lo from an FMA),
// e = y^2 x - 1 = fma(lo, x, fma(hi, x, -1)) to within 2^-46, and
// y sqrt(x) - 1 = e/2 - e^2/8 + ..., so |e|/2 is the relative error to
// within 2^-44.  out[3], out[4]: max relative error against the real result
// of rcp (|r x - 1|, exact in double) and of sqrt (|s - sqrt(x)| / sqrt(x),
// sqrt(x) in double), in units of 2^-30, rounded up.
__global__ void probe_kernel(unsigned int* out) {
  const uint64_t lo = 0x00800000ull, hi = 0x7F800000ull;
  unsigned int worst_r = 0, worst_s = 0, worst_q = 0, rel_r = 0, rel_s = 0;
  for (uint64_t b = lo + blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; b < hi;
       b += (uint64_t)gridDim.x * blockDim.x) {
    const float x = __uint_as_float((uint32_t)b);
    const float ra = rcp_apx(x), re = __frcp_rn(x);
    const float sa = sqrt_apx(x), se = __fsqrt_rn(x);
    if (re >= 1.17549435e-38f) {  // normal reciprocal (ftz flushes the rest)
      const int d = (int)__float_as_uint(ra) - (int)__float_as_uint(re);
      worst_r = max(worst_r, (unsigned int)abs(d));
      const double er = fabs((double)ra * (double)x - 1.0);
      rel_r = max(rel_r, (unsigned int)ceil(er * 1073741824.0));
    }
    const int ds = (int)__float_as_uint(sa) - (int)__float_as_uint(se);
    worst_s = max(worst_s, (unsigned int)abs(ds));
    const double sx = sqrt((double)x);
    rel_s = max(rel_s, (unsigned int)ceil(fabs((double)sa - sx) / sx * 1073741824.0));
    const float y = rsqrt_apx(x);
    const float hi = __fmul_rn(y, y);
    const float lo = __fmaf_rn(y, y, -hi);
    const float e = __fmaf_rn(lo, x, __fmaf_rn(hi, x, -1.0f));
    // relative error in units of 2^-24, rounded up after a small guard for
    // the evaluation's own error
    worst_q = max(worst_q, (unsigned int)ceilf(fabsf(e) * 0.5f * 16777216.0f + 0.01f));
  }
  atomicMax(out + 0, worst_r);
  atomicMax(out + 1, worst_s);
  atomicMax(out + 2, worst_q);
  atomicMax(out + 3, rel_r);
  atomicMax(out + 4, rel_s);
}

extern "C" int approx_probe(unsigned int* host_out) {
  unsigned int* d = nullptr;
  if (cudaMalloc(&d, 5 * sizeof(unsigned int)) != cudaSuccess) return 1;
  cudaMemset(d, 0, 5 * sizeof(unsigned int));
  probe_kernel<<<152 * 16, 256>>>(d);
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(host_out, d, 5 * sizeof(unsigned int), cudaMemcpyDeviceToHost);
  cudaFree(d);
  return e == cudaSuccess ? 0 : 2;
}
