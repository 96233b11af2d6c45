// Test helper: issue rates of the units the softmax leans on, measured per SM
// in clock cycles (clock64 around a long loop of independent operations; one
// CTA of 32 warps per SM). Kinds: 0 = ex2.approx.ftz.f32 (MUFU),
// 1 = ex2.approx.f16x2 (MUFU, two results per op), 2 = fma.rn.f32 (FMA pipe),
// 3 = fma.rn.f32x2 (packed FMA, two results per op).
#include <cstdint>

template <int KIND>
__global__ void __launch_bounds__(1024, 1) rate_kernel(int iters, float seed, float* sink, long long* cycles) {
  float a[8];
  uint32_t h[8];
  uint64_t p[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    a[j] = seed * (j + 1) * 1e-3f - 0.5f;
    h[j] = 0x3c003c00u ^ j;
    asm("mov.b64 %0, {%1, %2};" : "=l"(p[j]) : "f"(a[j]), "f"(a[j] * 0.5f));
  }
  const float m = 0.999f, c = 1e-4f;
  uint64_t m2, c2;
  asm("mov.b64 %0, {%1, %1};" : "=l"(m2) : "f"(m));
  asm("mov.b64 %0, {%1, %1};" : "=l"(c2) : "f"(c));
  __syncthreads();
  long long t0 = clock64();
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (KIND == 0) asm volatile("ex2.approx.ftz.f32 %0, %0;" : "+f"(a[j]));
      if (KIND == 1) asm volatile("ex2.approx.f16x2 %0, %0;" : "+r"(h[j]));
      if (KIND == 2) asm volatile("fma.rn.f32 %0, %0, %1, %2;" : "+f"(a[j]) : "f"(m), "f"(c));
      if (KIND == 3) asm volatile("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(p[j]) : "l"(m2), "l"(c2));
    }
  }
  __syncthreads();
  long long t1 = clock64();
  float acc = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) acc += a[j] + (float)(h[j] & 0xff) + (float)(p[j] & 0xff);
  if (acc == 12345.678f) sink[threadIdx.x] = acc;   // keeps the loops alive
  if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
}

// Operations per SM per clock cycle: result = ops / cycles (per CTA, averaged).
extern "C" double unit_rate(int kind, int sms, int iters) {
  float* sink = nullptr;
  long long* cyc = nullptr;
  cudaMalloc(&sink, 1024 * sizeof(float));
  cudaMalloc(&cyc, sms * sizeof(long long));
  switch (kind) {
    case 0: rate_kernel<0><<<sms, 1024>>>(iters, 1.f, sink, cyc); break;
    case 1: rate_kernel<1><<<sms, 1024>>>(iters, 1.f, sink, cyc); break;
    case 2: rate_kernel<2><<<sms, 1024>>>(iters, 1.f, sink, cyc); break;
    default: rate_kernel<3><<<sms, 1024>>>(iters, 1.f, sink, cyc); break;
  }
  long long host[1024];
  double rate = -1.0;
  if (cudaDeviceSynchronize() == cudaSuccess &&
      cudaMemcpy(host, cyc, sms * sizeof(long long), cudaMemcpyDeviceToHost) == cudaSuccess) {
    double mean = 0;
    for (int i = 0; i < sms; ++i) mean += (double)host[i] / sms;
    const double ops = 1024.0 * 8.0 * iters;   // instructions per CTA (= per SM)
    rate = ops / mean;
  }
  cudaFree(sink);
  cudaFree(cyc);
  return rate;
}
