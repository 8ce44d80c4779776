// Which operations of the MMA-issuing warp stall behind its tcgen05.mma in flight?
// 512 MMAs (M=128, N=128, K=16, SS) issued by lane 0 of warp 0, an extra operation every 8.
#include <cstdio>
#include <cstdint>
#include "ptx.cuh"
using namespace vs;

__device__ __forceinline__ void named_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }
__device__ __forceinline__ void named_arrive(int id, int n) { asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory"); }

template <int OP>
__global__ void __launch_bounds__(128, 1) k(long long* out, int nmma, unsigned long long* sink, const int* gflag) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  __shared__ uint64_t bar, done_bar;
  __shared__ uint32_t tslot;
  __shared__ uint4 vec;
  for (int i = threadIdx.x; i < 65536 / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(sm)[i] = 0x3f803f80u;
  if (threadIdx.x < 32) {
    tmem_alloc(&tslot, 512);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_init(&done_bar, 1);
    vec = make_uint4(1, 2, 3, 4);
    fence_mbar_init();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) mbar_arrive(&done_bar);
  __syncthreads();
  const uint32_t tb = tslot;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nev = nmma / 8 - 1;
  if (warp == 0) {
    const uint32_t idesc = idesc_bf16(128, 128, false, false);
    const uint32_t a = smem_u32(sm), b = smem_u32(sm + 32768);
    unsigned long long acc = 0;
    const long long t0 = clock64();
    for (int i = 0; i < nmma; ++i) {
      if (i > 0 && i % 8 == 0) {
        if (OP == 1) { named_sync(1, 64); named_arrive(2, 64); }
        if (OP == 2) acc += *(volatile const int*)(gflag + (i & 7));
        if (OP == 4) __syncwarp();
        if (OP == 5) acc += __shfl_sync(0xffffffffu, (int)i, 3);
        if (OP == 6) {
          uint32_t x0, x1, x2, x3;
          asm volatile("ld.volatile.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(x0), "=r"(x1), "=r"(x2), "=r"(x3) : "r"(smem_u32(&vec)));
          acc += x0 + x3;
        }
        if (OP == 7) { if (lane == 1) acc += mbar_try_wait(&done_bar, 0) ? 1 : 0; __syncwarp(); }
        if (OP == 8) { if (lane == 0) acc += mbar_try_wait(&done_bar, 0) ? 1 : 0; __syncwarp(); }
      }
      if (lane == 0) {
        const uint32_t off = (i & 3) * 32;
        umma_ss(tb + (i & 1) * 128, sdesc_sw128(a + off, 16, 1024), sdesc_sw128(b + off, 16, 1024), idesc,
                i >= 2 ? 1u : 0u);
      }
      __syncwarp();
    }
    if (lane == 0) {
      umma_commit(&bar);
      const bool ok = mbar_wait(&bar, 0, 2000000000ull);
      out[blockIdx.x] = ok ? clock64() - t0 : -1;
    }
    if (acc == 12345) sink[0] = acc;
  } else if (warp == 1) {
    if (OP == 1)
      for (int j = 0; j < nev; ++j) {
        named_arrive(1, 64);
        named_sync(2, 64);
      }
    if (OP == 3) {  // another warp hammers shared memory meanwhile
      unsigned long long acc = 0;
      for (int j = 0; j < 20000; ++j) acc += mbar_try_wait(&done_bar, 0) ? 1 : 0;
      if (acc == 12345) sink[0] = acc;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x < 32) tmem_dealloc(tb, 512);
}

template <int OP>
void run(long long* d, unsigned long long* sink, const int* gf, const char* name) {
  const int smem = 65536 + 1024, n = 512;
  cudaFuncSetAttribute(k<OP>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  for (int r = 0; r < 2; ++r) k<OP><<<152, 128, smem>>>(d, n, sink, gf);
  cudaError_t e = cudaDeviceSynchronize();
  long long h[152];
  cudaMemcpy(h, d, sizeof(h), cudaMemcpyDeviceToHost);
  double s = 0; bool bad = false;
  for (int i = 0; i < 152; ++i) { s += h[i]; if (h[i] < 0) bad = true; }
  printf("%-52s %.1f cyc/MMA%s [%s]\n", name, s / 152 / n, bad ? " TIMEOUT" : "", cudaGetErrorString(e));
}

int main() {
  long long* d; unsigned long long* sink; int* gf;
  cudaMalloc(&d, 152 * 8); cudaMalloc(&sink, 8); cudaMalloc(&gf, 64); cudaMemset(gf, 0, 64);
  run<0>(d, sink, gf, "nothing (whole warp in the loop)");
  run<1>(d, sink, gf, "named barrier sync with another warp");
  run<2>(d, sink, gf, "volatile global load (L1 hit)");
  run<3>(d, sink, gf, "another warp polls an mbarrier meanwhile");
  run<4>(d, sink, gf, "__syncwarp");
  run<5>(d, sink, gf, "shfl_sync");
  run<6>(d, sink, gf, "16-byte shared load");
  run<7>(d, sink, gf, "try_wait by lane 1 of the issuing warp");
  run<8>(d, sink, gf, "try_wait by lane 0 (the issuing lane)");
  return 0;
}
