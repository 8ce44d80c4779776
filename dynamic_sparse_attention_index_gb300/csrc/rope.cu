// Rotate-half RoPE (and its adjoint) over a token-major [L][H][d] bf16 tensor.
//
// MTraining review, section "Vertical-Slash 稀疏模式": the expectation
// equation pairs channel i with i + d/2 at frequency theta_i.  For i < d/2
// and phi = t * theta_i:  y_i = c (x_i cos phi - x_{i+d/2} sin phi),
// y_{i+d/2} = c (x_{i+d/2} cos phi + x_i sin phi), c the YaRN temperature.
//
// One thread owns (token t, 8 consecutive channel pairs) and walks all H
// heads, so each angle is formed once per (t, i) and every access is a
// 16-byte vector (8 bf16).  The angle t * theta_i is reduced modulo 2 pi in
// 64-bit fixed point: with theta_i / (2 pi) held as a 0.64 fraction, the
// wrapping integer product t * frac_i is the angle's fraction of a turn,
// exact up to the fraction's rounding (t reaches 2^20, where an fp32 product
// would lose whole radians; fp64 arithmetic is slow on this GPU).  Its top
// 32 bits read as a signed integer give the angle in [-pi, pi); the sine and
// cosine are taken in fp32.
#include <cuda_bf16.h>

#include <cmath>
#include <cstring>

#include "common.cuh"

namespace vs {

__global__ void __launch_bounds__(256) rope_kernel(const __nv_bfloat16* x, __nv_bfloat16* y,
                                                   int L, int H, int d, int transpose, float mscale,
                                                   RopeArgs freqs) {
  if (freqs.skip_if != nullptr && *freqs.skip_if != 0) return;
  const int half = d >> 1, ng = half >> 3;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)L * ng) return;
  const int t = (int)(idx / ng);
  const int g = (int)(idx - (long long)t * ng);
  const float kTurnToRad = 1.4629180792671596e-09f;  // 2 pi / 2^32
  float cs[8], sn[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint64_t frac = (uint64_t)t * freqs.turn[8 * g + k];  // modulo 2^64: the fraction of a turn
    const float phi = (float)(int32_t)(uint32_t)(frac >> 32) * kTurnToRad;
    float s1, c1;
    sincosf(phi, &s1, &c1);
    if (transpose) s1 = -s1;
    cs[k] = c1 * mscale;
    sn[k] = s1 * mscale;
  }
  const size_t row = (size_t)t * H * d + 8 * g;
  for (int h = 0; h < H; ++h) {
    const size_t o = row + (size_t)h * d;
    const uint4 va = *reinterpret_cast<const uint4*>(x + o);
    const uint4 vb = *reinterpret_cast<const uint4*>(x + o + half);
    const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&va);
    const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&vb);
    uint4 ya, yb;
    __nv_bfloat162* qa = reinterpret_cast<__nv_bfloat162*>(&ya);
    __nv_bfloat162* qb = reinterpret_cast<__nv_bfloat162*>(&yb);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 a = __bfloat1622float2(pa[k]), b = __bfloat1622float2(pb[k]);
      const int k0 = 2 * k, k1 = 2 * k + 1;
      qa[k] = __floats2bfloat162_rn(a.x * cs[k0] - b.x * sn[k0], a.y * cs[k1] - b.y * sn[k1]);
      qb[k] = __floats2bfloat162_rn(b.x * cs[k0] + a.x * sn[k0], b.y * cs[k1] + a.y * sn[k1]);
    }
    *reinterpret_cast<uint4*>(y + o) = ya;
    *reinterpret_cast<uint4*>(y + o + half) = yb;
  }
}

void rope_fill(const vs_params& p, RopeArgs& a) {
  // theta_i = base^(-2i/d); YaRN NTK-by-parts: gamma_i = clip((r_i - 1)/(32 - 1), 0, 1),
  // r_i = orig_len * theta_i / (2 pi); theta'_i = theta_i (gamma_i + (1 - gamma_i)/s)
  const double s = p.yarn_factor;
  for (int i = 0; i < p.d / 2; ++i) {
    double f = std::pow(p.rope_theta, -2.0 * i / p.d);
    if (s > 1.0) {
      const double r = p.yarn_orig_len * f / (2.0 * 3.14159265358979323846);
      double g = (r - 1.0) / (32.0 - 1.0);
      g = g < 0.0 ? 0.0 : (g > 1.0 ? 1.0 : g);
      f = f * (g + (1.0 - g) / s);
    }
    // f / (2 pi) < 1; its double value scaled by 2^64 converts to uint64 exactly
    const double turns = f / (2.0 * 3.14159265358979323846);
    a.turn[i] = turns < 1.0 ? (uint64_t)(turns * 18446744073709551616.0) : ~0ull;
  }
  a.mscale = s > 1.0 ? (float)(0.1 * std::log(s) + 1.0) : 1.0f;
}

cudaError_t launch_rope(const RopeArgs& a, cudaStream_t s) {
  const long long n = (long long)a.L * (a.d / 16);
  const int threads = 256;
  const long long blocks = (n + threads - 1) / threads;
  rope_kernel<<<(unsigned)blocks, threads, 0, s>>>(static_cast<const __nv_bfloat16*>(a.x),
                                                   static_cast<__nv_bfloat16*>(a.y), a.L, a.H, a.d, a.transpose,
                                                   a.mscale, a);
  return cudaGetLastError();
}

cudaError_t launch_rope_adjoint(const vs_params& p, void* dQ, void* dK, const int32_t* dq_skip_if, cudaStream_t s) {
  RopeArgs a;
  std::memset(&a, 0, sizeof(a));
  a.L = p.L;
  a.d = p.d;
  a.transpose = 1;
  rope_fill(p, a);
  a.x = dK;
  a.y = dK;
  a.H = p.Hkv;
  cudaError_t e = launch_rope(a, s);
  if (e != cudaSuccess) return e;
  a.x = dQ;
  a.y = dQ;
  a.H = p.Hq;
  a.skip_if = dq_skip_if;
  return launch_rope(a, s);
}

}  // namespace vs
