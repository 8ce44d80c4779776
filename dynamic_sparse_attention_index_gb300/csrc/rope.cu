// Rotate-half RoPE (and its adjoint) over a token-major [L][H][d] bf16 tensor.
//
// MTraining review, section "Vertical-Slash 稀疏模式": the expectation
// equation pairs channel i with i + d/2 at frequency theta_i.  For i < d/2
// and phi = t * theta_i:  y_i = c (x_i cos phi - x_{i+d/2} sin phi),
// y_{i+d/2} = c (x_{i+d/2} cos phi + x_i sin phi), c the YaRN temperature.
//
// One thread owns (token t, channel pair i) and walks all H heads, so the
// angle is formed once per (t, i): the product t * theta_i and its reduction
// to [-pi, pi] are done in fp64 (t reaches 2^20, where an fp32 product would
// lose whole radians), the sine and cosine of the reduced angle in fp32.
#include <cuda_bf16.h>

#include "common.cuh"

namespace vs {

__global__ void __launch_bounds__(256) rope_kernel(const __nv_bfloat16* x, __nv_bfloat16* y,
                                                   int L, int H, int d, int transpose, float mscale,
                                                   RopeArgs freqs) {
  const int half = d >> 1;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)L * half) return;
  const int t = (int)(idx / half);
  const int i = (int)(idx - (long long)t * half);
  const double kTwoPi = 6.283185307179586476925286766559;
  double phi = (double)t * freqs.inv_freq[i];
  phi -= kTwoPi * rint(phi / kTwoPi);
  float sn, cs;
  sincosf((float)phi, &sn, &cs);
  if (transpose) sn = -sn;
  cs *= mscale;
  sn *= mscale;
  const size_t row = (size_t)t * H * d;
  for (int h = 0; h < H; ++h) {
    const size_t o = row + (size_t)h * d + i;
    const float a = __bfloat162float(x[o]);
    const float b = __bfloat162float(x[o + half]);
    y[o] = __float2bfloat16_rn(a * cs - b * sn);
    y[o + half] = __float2bfloat16_rn(b * cs + a * sn);
  }
}

cudaError_t launch_rope(const RopeArgs& a, cudaStream_t s) {
  const long long n = (long long)a.L * (a.d / 2);
  const int threads = 256;
  const long long blocks = (n + threads - 1) / threads;
  rope_kernel<<<(unsigned)blocks, threads, 0, s>>>(static_cast<const __nv_bfloat16*>(a.x),
                                                   static_cast<__nv_bfloat16*>(a.y), a.L, a.H, a.d, a.transpose,
                                                   a.mscale, a);
  return cudaGetLastError();
}

}  // namespace vs
