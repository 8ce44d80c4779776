// tcgen05 pipe probe: (1) M=128 N=128 TS vs SS rate, (2) how far the issuing thread runs ahead
// of execution (issue-loop time vs completion), (3) cost of a commit on a busy pipe
#include <cstdio>
#include <cstdint>
#include "ptx.cuh"
using namespace vs;

template <bool TS>
__global__ void __launch_bounds__(128, 1) k(long long* out, int nmma, int ncommit_every) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  __shared__ uint64_t bar, cbar;
  __shared__ uint32_t tslot;
  for (int i = threadIdx.x; i < 65536 / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(sm)[i] = 0x3f803f80u;
  if (threadIdx.x < 32) {
    tmem_alloc(&tslot, 512);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_init(&cbar, 1);
    fence_mbar_init();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tslot;
  if (threadIdx.x == 0) {
    const uint32_t idesc = idesc_bf16(128, 128, false, TS);
    const uint32_t a = smem_u32(sm), b = smem_u32(sm + 32768);
    long long tc = 0;
    const long long t0 = clock64();
    for (int i = 0; i < nmma; ++i) {
      if (ncommit_every && i > 0 && i % ncommit_every == 0) {
        const long long c0 = clock64();
        umma_commit(&cbar);
        tc += clock64() - c0;
      }
      const uint32_t off = (i & 3) * 32;
      const uint32_t d = tb + (i & 1) * 128;
      if (TS)
        umma_ts(d, tb + 256 + (i & 3) * 8, sdesc_sw128(b + (i & 3) * 2048, 16, 1024), idesc, i >= 2 ? 1u : 0u);
      else
        umma_ss(d, sdesc_sw128(a + off, 16, 1024), sdesc_sw128(b + off, 16, 1024), idesc, i >= 2 ? 1u : 0u);
    }
    const long long t1 = clock64();
    umma_commit(&bar);
    const bool ok = mbar_wait(&bar, 0, 2000000000ull);
    const long long t2 = clock64();
    out[blockIdx.x * 3] = ok ? t1 - t0 : -1;
    out[blockIdx.x * 3 + 1] = ok ? t2 - t0 : -1;
    out[blockIdx.x * 3 + 2] = tc;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x < 32) tmem_dealloc(tb, 512);
}

template <bool TS>
void run(long long* d, int nmma, int ce) {
  const int smem = 65536 + 1024;
  cudaFuncSetAttribute(k<TS>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  for (int r = 0; r < 2; ++r) k<TS><<<152, 128, smem>>>(d, nmma, ce);
  cudaError_t e = cudaDeviceSynchronize();
  long long h[152 * 3];
  cudaMemcpy(h, d, sizeof(h), cudaMemcpyDeviceToHost);
  double s0 = 0, s1 = 0, s2 = 0;
  bool bad = false;
  for (int i = 0; i < 152; ++i) {
    if (h[3 * i] < 0) bad = true;
    s0 += h[3 * i]; s1 += h[3 * i + 1]; s2 += h[3 * i + 2];
  }
  const int nc = ce ? (nmma - 1) / ce : 0;
  printf("M=128 N=128 %s n=%4d commit/%d: issue loop %.0f cyc, done %.0f cyc (%.1f cyc/MMA), commit %.1f cyc each%s [%s]\n",
         TS ? "TS" : "SS", nmma, ce, s0 / 152, s1 / 152, s1 / 152 / nmma, nc ? s2 / 152 / nc : 0.0, bad ? " TIMEOUT" : "",
         cudaGetErrorString(e));
}

int main() {
  long long* d;
  cudaMalloc(&d, 152 * 3 * 8);
  for (int n : {1, 2, 4, 8, 16, 32, 512}) run<false>(d, n, 0);
  for (int n : {1, 2, 4, 8, 16, 32, 512}) run<true>(d, n, 0);
  run<false>(d, 512, 8);
  run<true>(d, 512, 8);
  run<false>(d, 512, 4);
  return 0;
}
