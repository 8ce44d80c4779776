// Cost of tcgen05.commit (no MMA in flight): bursts, commit->observed latency, and smem atomics
#include <cstdio>
#include <cstdint>
#include "ptx.cuh"
using namespace vs;

template <int OP>
__global__ void __launch_bounds__(64, 1) k(long long* out, int n) {
  __shared__ uint64_t bar[4];
  __shared__ unsigned long long cnt[4];
  __shared__ uint32_t tslot;
  if (threadIdx.x < 32) {
    tmem_alloc(&tslot, 32);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < 4; ++i) { mbar_init(&bar[i], 1); cnt[i] = 0; }
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tslot;
  if (threadIdx.x == 0) {
    bool ok = true;
    const long long t0 = clock64();
    for (int i = 0; i < n && ok; ++i) {
      if (OP == 0) umma_commit(&bar[0]);                       // burst of commits, nobody waits
      if (OP == 1) { umma_commit(&bar[0]); umma_commit(&bar[1]); umma_commit(&bar[2]); umma_commit(&bar[3]); }
      if (OP == 2) {                                            // commit then wait for its arrival
        umma_commit(&bar[0]);
        const long long c0 = clock64();
        while (!mbar_try_wait(&bar[0], i & 1)) if (clock64() - c0 > 1000000000ll) { ok = false; break; }
      }
      if (OP == 3) atomicAdd(&cnt[i & 3], 1ull);                // shared 64-bit atomics
      if (OP == 4) mbar_arrive(&bar[0]);                        // plain arrive
    }
    out[blockIdx.x] = ok ? clock64() - t0 : -1;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x < 32) tmem_dealloc(tb, 32);
}

template <int OP>
void run(long long* d, const char* name, int per) {
  const int n = 4096;
  for (int r = 0; r < 2; ++r) k<OP><<<152, 64>>>(d, n);
  cudaError_t e = cudaDeviceSynchronize();
  long long h[152];
  cudaMemcpy(h, d, sizeof(h), cudaMemcpyDeviceToHost);
  double s = 0; bool bad = false;
  for (int i = 0; i < 152; ++i) { s += h[i]; if (h[i] < 0) bad = true; }
  printf("%-40s %.1f cycles each%s [%s]\n", name, s / 152 / n / per, bad ? " TIMEOUT" : "", cudaGetErrorString(e));
}

int main() {
  long long* d;
  cudaMalloc(&d, 152 * 8);
  run<0>(d, "commit burst (one barrier)", 1);
  run<1>(d, "commit burst (four barriers)", 4);
  run<2>(d, "commit + wait for its arrival", 1);
  run<3>(d, "shared atomicAdd u64", 1);
  run<4>(d, "mbarrier.arrive", 1);
  return 0;
}
