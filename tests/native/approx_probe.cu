// approx_probe.cu -- test helper: worst-case error, in units in the last
// place, of the hardware approximations the step kernel certifies
// (rcp.approx.ftz.f32, sqrt.approx.ftz.f32) against the correctly rounded
// IEEE results, over every positive normal fp32 input.
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

// inputs: bits in [0x00800000, 0x7F800000) (all positive normals); one thread
// per input, grid-stride.  out[0] = max ulp error of rcp, out[1] = of sqrt.
__global__ void probe_kernel(unsigned int* out) {
  const uint64_t lo = 0x00800000ull, hi = 0x7F800000ull;
  unsigned int worst_r = 0, worst_s = 0;
  for (uint64_t b = lo + blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; b < hi;
       b += (uint64_t)gridDim.x * blockDim.x) {
    const float x = __uint_as_float((uint32_t)b);
    const float ra = rcp_apx(x), re = __frcp_rn(x);
    const float sa = sqrt_apx(x), se = __fsqrt_rn(x);
    if (re >= 1.17549435e-38f) {  // normal reciprocal (ftz flushes the rest)
      const int d = (int)__float_as_uint(ra) - (int)__float_as_uint(re);
      worst_r = max(worst_r, (unsigned int)abs(d));
    }
    const int ds = (int)__float_as_uint(sa) - (int)__float_as_uint(se);
    worst_s = max(worst_s, (unsigned int)abs(ds));
  }
  atomicMax(out + 0, worst_r);
  atomicMax(out + 1, worst_s);
}

extern "C" int approx_probe(unsigned int* host_out) {
  unsigned int* d = nullptr;
  if (cudaMalloc(&d, 2 * sizeof(unsigned int)) != cudaSuccess) return 1;
  cudaMemset(d, 0, 2 * sizeof(unsigned int));
  probe_kernel<<<152 * 16, 256>>>(d);
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(host_out, d, 2 * sizeof(unsigned int), cudaMemcpyDeviceToHost);
  cudaFree(d);
  return e == cudaSuccess ? 0 : 2;
}
