// Which MMA-thread operations between tcgen05.mma issues stall the tensor pipe?
// 512 MMAs (M=128, N=128, K=16, SS) with an extra operation every 8.
#include <cstdio>
#include <cstdint>
#include "ptx.cuh"
using namespace vs;

template <int OP>
__global__ void __launch_bounds__(128, 1) k(long long* out, int nmma, unsigned long long* sink) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  __shared__ uint64_t bar, cbar, done_bar;
  __shared__ uint32_t tslot;
  __shared__ volatile int flag;
  for (int i = threadIdx.x; i < 65536 / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(sm)[i] = 0x3f803f80u;
  if (threadIdx.x < 32) {
    tmem_alloc(&tslot, 512);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_init(&cbar, 1);
    mbar_init(&done_bar, 1);
    flag = 0;
    fence_mbar_init();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) mbar_arrive(&done_bar);  // phase 0 of done_bar complete
  __syncthreads();
  const uint32_t tb = tslot;
  if (threadIdx.x == 0) {
    const uint32_t idesc = idesc_bf16(128, 128, false, false);
    const uint32_t a = smem_u32(sm), b = smem_u32(sm + 32768);
    unsigned long long acc = 0;
    const long long t0 = clock64();
    for (int i = 0; i < nmma; ++i) {
      if (i > 0 && i % 8 == 0) {
        if (OP == 1) umma_commit(&cbar);
        if (OP == 2) acc += clock64();
        if (OP == 3) { umma_commit(&cbar); acc += clock64(); }
        if (OP == 4) acc += mbar_try_wait(&done_bar, 0) ? 1 : 0;
        if (OP == 5) acc += mbar_test_wait(&done_bar, 0) ? 1 : 0;
        if (OP == 6) acc += flag;
        if (OP == 7) tc_fence_after();
        if (OP == 8) { umma_commit(&cbar); acc += mbar_try_wait(&done_bar, 0) ? 1 : 0; tc_fence_after(); }
        if (OP == 9) acc += mbar_wait(&done_bar, 0, 1000000000ull) ? 1 : 0;
        if (OP == 10) { acc += clock64(); acc += mbar_try_wait(&done_bar, 0) ? 1 : 0; }
        if (OP == 11) { for (int j = 0; j < (1 << 20); ++j) if (mbar_try_wait(&done_bar, 0)) { acc += j; break; } }
        if (OP == 12) acc += mbar_try_wait_sleep(&done_bar, 0, 100000u) ? 1 : 0;
        if (OP == 13) { for (int j = 0; j < (1 << 20); ++j) if (mbar_test_wait(&done_bar, 0)) { acc += j; break; } }
      }
      const uint32_t off = (i & 3) * 32;
      umma_ss(tb + (i & 1) * 128, sdesc_sw128(a + off, 16, 1024), sdesc_sw128(b + off, 16, 1024), idesc, i >= 2 ? 1u : 0u);
    }
    umma_commit(&bar);
    const bool ok = mbar_wait(&bar, 0, 2000000000ull);
    out[blockIdx.x] = ok ? clock64() - t0 : -1;
    if (acc == 12345) sink[0] = acc;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x < 32) tmem_dealloc(tb, 512);
}

template <int OP>
void run(long long* d, unsigned long long* sink, const char* name) {
  const int smem = 65536 + 1024, n = 512;
  cudaFuncSetAttribute(k<OP>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  for (int r = 0; r < 2; ++r) k<OP><<<152, 128, smem>>>(d, n, sink);
  cudaError_t e = cudaDeviceSynchronize();
  long long h[152];
  cudaMemcpy(h, d, sizeof(h), cudaMemcpyDeviceToHost);
  double s = 0; bool bad = false;
  for (int i = 0; i < 152; ++i) { s += h[i]; if (h[i] < 0) bad = true; }
  printf("%-44s %.1f cyc/MMA%s [%s]\n", name, s / 152 / n, bad ? " TIMEOUT" : "", cudaGetErrorString(e));
}

int main() {
  long long* d; unsigned long long* sink;
  cudaMalloc(&d, 152 * 8); cudaMalloc(&sink, 8);
  run<0>(d, sink, "nothing");
  run<1>(d, sink, "commit");
  run<2>(d, sink, "clock64");
  run<3>(d, sink, "commit + clock64");
  run<4>(d, sink, "try_wait (complete phase)");
  run<5>(d, sink, "test_wait (complete phase)");
  run<6>(d, sink, "volatile smem load");
  run<7>(d, sink, "tcgen05.fence::after_thread_sync");
  run<8>(d, sink, "commit + try_wait + fence");
  run<9>(d, sink, "mbar_wait helper (complete phase)");
  run<10>(d, sink, "clock64 + try_wait");
  run<11>(d, sink, "bounded try_wait loop (complete phase)");
  run<12>(d, sink, "try_wait with suspend hint (complete phase)");
  run<13>(d, sink, "bounded test_wait loop (complete phase)");
  return 0;
}
