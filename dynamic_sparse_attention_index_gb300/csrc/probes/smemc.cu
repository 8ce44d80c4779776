// Shared-memory contention between tcgen05.mma operand reads and other warps.
// Warp 0 lane 0 streams 512 MMAs (M=128, N=128, K=16; SS or TS); warps 1-3 meanwhile
// (a) time dependent 4-byte shared loads, or (b) store 16 B per thread per iteration.
#include <cstdio>
#include <cstdint>
#include "ptx.cuh"
using namespace vs;

template <int OP, bool TS, bool MMA>
__global__ void __launch_bounds__(128, 1) k(long long* out, int nmma, unsigned long long* sink) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  __shared__ uint64_t bar;
  __shared__ uint32_t tslot;
  __shared__ int chase[1024];
  __shared__ volatile int go;
  for (int i = threadIdx.x; i < 98304 / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(sm)[i] = 0x3f803f80u;
  for (int i = threadIdx.x; i < 1024; i += blockDim.x) chase[i] = (i * 97 + 13) & 1023;
  if (threadIdx.x < 32) {
    tmem_alloc(&tslot, 512);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    go = 0;
    fence_mbar_init();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tslot;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(128, 128, false, TS);
      const uint32_t a = smem_u32(sm), b = smem_u32(sm + 32768);
      go = 1;
      const long long t0 = clock64();
      if (MMA) {
        for (int i = 0; i < nmma; ++i) {
          const uint32_t off = (i & 3) * 32;
          if (TS)
            umma_ts(tb + (i & 1) * 128, tb + 256 + (i & 3) * 8, sdesc_sw128(b + (i & 3) * 2048, 16, 1024), idesc,
                    i >= 2 ? 1u : 0u);
          else
            umma_ss(tb + (i & 1) * 128, sdesc_sw128(a + off, 16, 1024), sdesc_sw128(b + off, 16, 1024), idesc,
                    i >= 2 ? 1u : 0u);
        }
      } else {
        while (clock64() - t0 < 33000) {
        }
      }
      umma_commit(&bar);
      const bool ok = mbar_wait(&bar, 0, 2000000000ull);
      out[blockIdx.x * 2] = ok ? clock64() - t0 : -1;
      go = 2;
    }
  } else {
    // other warps: work until the MMA stream ends (bounded)
    for (int sp = 0; sp < (1 << 24) && go == 0; ++sp) {
    }
    long long n = 0, tsum = 0;
    int idx = threadIdx.x & 1023;
    uint8_t* dst = sm + 65536 + (threadIdx.x - 32) * 16;
    for (int it = 0; it < 100000 && go == 1; ++it) {
      if (OP == 0) {
        const long long c0 = clock64();
#pragma unroll
        for (int j = 0; j < 8; ++j) idx = chase[idx];
        tsum += clock64() - c0;
        n += 8;
      } else {
        const long long c0 = clock64();
#pragma unroll
        for (int j = 0; j < 8; ++j)
          asm volatile("st.volatile.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(smem_u32(dst + (j & 1) * 1536)),
                       "r"(idx), "r"(j), "r"(it), "r"(0) : "memory");
        tsum += clock64() - c0;
        n += 8;
      }
    }
    if (threadIdx.x == 32) out[blockIdx.x * 2 + 1] = n ? (tsum * 100) / n : -1;
    if (idx == 123456) sink[0] = idx;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x < 32) tmem_dealloc(tb, 512);
}

template <int OP, bool TS, bool MMA>
void run(long long* d, unsigned long long* sink, const char* name) {
  const int smem = 98304 + 1024, n = 512;
  cudaFuncSetAttribute(k<OP, TS, MMA>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  for (int r = 0; r < 2; ++r) k<OP, TS, MMA><<<152, 128, smem>>>(d, n, sink);
  cudaError_t e = cudaDeviceSynchronize();
  long long h[304];
  cudaMemcpy(h, d, sizeof(h), cudaMemcpyDeviceToHost);
  double s0 = 0, s1 = 0;
  for (int i = 0; i < 152; ++i) { s0 += h[2 * i]; s1 += h[2 * i + 1]; }
  printf("%-48s MMA %.1f cyc/MMA, other warps %.2f cyc per access [%s]\n", name, s0 / 152 / n, s1 / 152 / 100.0,
         cudaGetErrorString(e));
}

int main() {
  long long* d; unsigned long long* sink;
  cudaMalloc(&d, 304 * 8); cudaMalloc(&sink, 8);
  run<0, false, false>(d, sink, "no MMA, dependent 4-byte loads");
  run<0, false, true>(d, sink, "SS MMA stream, dependent 4-byte loads");
  run<0, true, true>(d, sink, "TS MMA stream, dependent 4-byte loads");
  run<1, false, false>(d, sink, "no MMA, 16-byte stores (3 warps)");
  run<1, false, true>(d, sink, "SS MMA stream, 16-byte stores (3 warps)");
  run<1, true, true>(d, sink, "TS MMA stream, 16-byte stores (3 warps)");
  return 0;
}
