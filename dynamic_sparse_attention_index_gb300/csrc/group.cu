// GQA-group-shared sparse index: every query head of a key/value group uses
// the union of the group's per-head selections.
//
// MTraining review, section 三/核心创新/2 "分布式稀疏索引近似" (kernel-aware
// approximation granularity: a coarser index costs less to use but keeps
// more redundant entries).  With one index per group, the G query heads
// that share a key/value head also share every vertical line and slash band,
// so a key block is active for the same query blocks of all G heads.  The
// union keeps every line any head of the group selected, so each head's
// recall is at least that of its own selection; the price is density.
#include "common.cuh"

namespace vs {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;

// block-wide exclusive scan of one int per thread; returns the total
__device__ int block_scan(int x, int* excl, int* wsum) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = x;
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  int before = 0, total = 0;
  for (int k = 0; k < kWarps; ++k) {
    if (k < warp) before += wsum[k];
    total += wsum[k];
  }
  __syncthreads();
  *excl = before + incl - x;
  return total;
}

// One CTA per key/value group.  Shared memory: vertical bitmap (L bits),
// kept-band flags (nbs bytes), notS[nbs] = #{B in [1, x] not kept}.
__global__ void __launch_bounds__(kThreads, 1)
    group_union_kernel(int L, int Hq, int G, int bs, int32_t* v_idx, int32_t* v_cnt, int32_t* s_idx,
                       int32_t* s_cnt, int64_t* active) {
  extern __shared__ uint8_t sm[];
  const int nbs = L / bs;
  const int nwl = L / 32;
  uint32_t* vb = reinterpret_cast<uint32_t*>(sm);
  uint8_t* inS = sm + (size_t)nwl * 4;
  int32_t* notS = reinterpret_cast<int32_t*>(inS + align_up((size_t)nbs, 16));
  __shared__ int wsum[kWarps];
  __shared__ int carry_s;
  __shared__ unsigned long long red[kWarps];
  const int grp = blockIdx.x;
  const int h0 = grp * G;
  for (int w = threadIdx.x; w < nwl; w += kThreads) vb[w] = 0u;
  for (int B = threadIdx.x; B < nbs; B += kThreads) inS[B] = B == 0 ? 1 : 0;
  __syncthreads();
  // the union of the group's sets (every head is read before any is written)
  for (int hh = 0; hh < G; ++hh) {
    const int h = h0 + hh;
    const int nv = v_cnt[h], ns = s_cnt[h];
    for (int j = threadIdx.x; j < nv; j += kThreads) {
      const int m = v_idx[(size_t)h * L + j];
      if (m >= 0 && m < L) atomicOr(&vb[m >> 5], 1u << (m & 31));
    }
    for (int j = threadIdx.x; j < ns; j += kThreads) {
      const int B = s_idx[(size_t)h * nbs + j];
      if (B >= 0 && B < nbs) inS[B] = 1;
    }
  }
  __syncthreads();

  // kept bands in ascending order, their entries, and notS
  if (threadIdx.x == 0) carry_s = 0;
  __syncthreads();
  unsigned long long slash_e = 0;
  for (int base = 0; base < nbs; base += kThreads) {
    const int B = base + threadIdx.x;
    const int k = (B < nbs && inS[B]) ? 1 : 0;
    const int nk = (B < nbs && B >= 1 && !inS[B]) ? 1 : 0;
    int pos, pos_nk;
    const int tot = block_scan(k, &pos, wsum);
    const int tot_nk = block_scan(nk, &pos_nk, wsum);
    const int c0 = carry_s;
    if (B < nbs) {
      // notS[B] counts the not-kept bands 1..B: the carried count of earlier
      // chunks (stored in notS[base - 1]) plus this chunk's inclusive scan
      const int prev = base > 0 ? notS[base - 1] : 0;
      notS[B] = prev + pos_nk + nk;
      if (k) {
        for (int hh = 0; hh < G; ++hh) s_idx[(size_t)(h0 + hh) * nbs + c0 + pos] = B;
        slash_e += B == 0 ? (unsigned long long)nbs * (unsigned long long)(bs * (bs + 1) / 2)
                          : (unsigned long long)(nbs - B) * (unsigned long long)bs * (unsigned long long)bs;
      }
    }
    (void)tot_nk;
    __syncthreads();
    if (threadIdx.x == 0) carry_s = c0 + tot;
    __syncthreads();
  }
  const int ns = carry_s;
  __syncthreads();

  // kept verticals in ascending order and their entries outside kept bands
  if (threadIdx.x == 0) carry_s = 0;
  __syncthreads();
  unsigned long long vert_e = 0;
  for (int base = 0; base < nwl; base += kThreads) {
    const int w = base + threadIdx.x;
    const uint32_t u = w < nwl ? vb[w] : 0u;
    int pos;
    const int tot = block_scan(__popc(u), &pos, wsum);
    const int c0 = carry_s;
    uint32_t x = u;
    int q = c0 + pos;
    while (x) {
      const int bit = __ffs(x) - 1;
      x &= x - 1;
      const int m = w * 32 + bit;
      for (int hh = 0; hh < G; ++hh) v_idx[(size_t)(h0 + hh) * L + q] = m;
      vert_e += (unsigned long long)bs * (unsigned long long)notS[nbs - 1 - m / bs];
      ++q;
    }
    __syncthreads();
    if (threadIdx.x == 0) carry_s = c0 + tot;
    __syncthreads();
  }
  const int nv = carry_s;

  // exact active entries of each head of the group (all equal)
  unsigned long long e = slash_e + vert_e;
  for (int o = 16; o > 0; o >>= 1) e += __shfl_xor_sync(0xffffffffu, e, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = e;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long t = 0;
    for (int k = 0; k < kWarps; ++k) t += red[k];
    for (int hh = 0; hh < G; ++hh) {
      v_cnt[h0 + hh] = nv;
      s_cnt[h0 + hh] = ns;
      if (active) active[h0 + hh] = (int64_t)t;
    }
  }
}

}  // namespace

size_t group_union_smem_bytes(int L, int bs) {
  const size_t nbs = (size_t)L / bs;
  return (size_t)(L / 32) * 4 + align_up(nbs, 16) + nbs * 4;
}

cudaError_t launch_group_union(const vs_params& p, const vs_index& ix, cudaStream_t s) {
  const int bs = kBlock * p.stripes;
  const size_t smem = group_union_smem_bytes(p.L, bs);
  cudaError_t e = cudaFuncSetAttribute(group_union_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  group_union_kernel<<<p.Hkv, kThreads, smem, s>>>(p.L, p.Hq, p.Hq / p.Hkv, bs, ix.v_idx, ix.v_cnt, ix.s_idx,
                                                   ix.s_cnt, ix.active_entries);
  return cudaGetLastError();
}

}  // namespace vs
