// MMA batches of 8 (M=128, N=128, K=16, SS) issued by lane 0 of warp 0; between batches a hand-off
// with warp 1 (the scheduler), which does nothing else.  Does the hand-off slow the MMAs?
#include <cstdio>
#include <cstdint>
#include "ptx.cuh"
using namespace vs;

__device__ __forceinline__ uint32_t red_popc(uint32_t id, uint32_t n, bool pred) {
  uint32_t r;
  asm volatile("{\n .reg .pred p;\n setp.ne.u32 p, %3, 0;\n bar.red.popc.u32 %0, %1, %2, p;\n}\n"
               : "=r"(r) : "r"(id), "r"(n), "r"((uint32_t)pred) : "memory");
  return r;
}
__device__ __forceinline__ void nsync(uint32_t id, uint32_t n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }
__device__ __forceinline__ void narrive(uint32_t id, uint32_t n) { asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory"); }

template <int OP>
__global__ void __launch_bounds__(128, 1) k(long long* out, int nb, unsigned long long* sink) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  __shared__ uint64_t bar;
  __shared__ uint32_t tslot;
  for (int i = threadIdx.x; i < 65536 / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(sm)[i] = 0x3f803f80u;
  if (threadIdx.x < 32) {
    tmem_alloc(&tslot, 512);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tslot;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned long long acc = 0;
  if (warp == 0) {
    const uint32_t idesc = idesc_bf16(128, 128, false, false);
    const uint32_t a = smem_u32(sm), b = smem_u32(sm + 32768);
    const long long t0 = clock64();
    for (int j = 0; j < nb; ++j) {
      if (OP == 1) acc += red_popc(1, 64, false);
      if (OP == 2) { nsync(1, 64); narrive(2, 64); }
      if (lane == 0) {
        tc_fence_after();
        for (int i = 0; i < 8; ++i) {
          const uint32_t off = (i & 3) * 32;
          umma_ss(tb + (j & 1) * 128, sdesc_sw128(a + off, 16, 1024), sdesc_sw128(b + off, 16, 1024), idesc,
                  i > 0 ? 1u : 0u);
        }
        umma_commit(&bar);
      }
      __syncwarp();
    }
    if (lane == 0) {
      // the last commit's phase: nb completions in all, parity of the last one
      const bool ok = mbar_wait(&bar, (nb - 1) & 1, 2000000000ull);
      out[blockIdx.x] = ok ? clock64() - t0 : -1;
    }
  } else if (warp == 1) {
    for (int j = 0; j < nb; ++j) {
      if (OP == 1) acc += red_popc(1, 64, lane < 5);
      if (OP == 2) { narrive(1, 64); nsync(2, 64); }
    }
  }
  if (acc == 123456789) sink[0] = acc;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x < 32) tmem_dealloc(tb, 512);
}

template <int OP>
void run(long long* d, unsigned long long* sink, const char* name) {
  const int smem = 65536 + 1024, nb = 64;
  cudaFuncSetAttribute(k<OP>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  for (int r = 0; r < 2; ++r) k<OP><<<152, 128, smem>>>(d, nb, sink);
  cudaError_t e = cudaDeviceSynchronize();
  long long h[152];
  cudaMemcpy(h, d, sizeof(h), cudaMemcpyDeviceToHost);
  double s = 0; bool bad = false;
  for (int i = 0; i < 152; ++i) { s += h[i]; if (h[i] < 0) bad = true; }
  printf("%-44s %.1f cyc/MMA%s [%s]\n", name, s / 152 / (nb * 8), bad ? " TIMEOUT" : "", cudaGetErrorString(e));
}

int main() {
  long long* d; unsigned long long* sink;
  cudaMalloc(&d, 152 * 8); cudaMalloc(&sink, 8);
  run<0>(d, sink, "batches of 8, no hand-off");
  run<1>(d, sink, "batches of 8, bar.red.popc hand-off");
  run<2>(d, sink, "batches of 8, bar.sync / bar.arrive ping-pong");
  return 0;
}
