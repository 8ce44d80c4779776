// Anti-diagonal block scorer: an alternative sparse index (the ablation row
// "MTraining w/ XAttn Idx." of the MTraining review, section 五 "实验结果",
// table "训练效率结果"; the pages name the scorer only, and the reading here
// is the published XAttention block scorer).
//
// Per query head, with stride S: strided row r is the query group of tokens
// rS .. rS+S-1 and strided column c the key group cS .. cS+S-1; cell (r, c)
// is scored by the mean scaled logit on the anti-diagonal of that S x S
// sub-block,
//     z[r, c] = scale / S * sum_j q[rS + j] . k[cS + S-1-j],
// cells c > r are masked, P is the softmax of z over each strided row, and
// the block score of block row I, block column J (bs-token blocks, bs / S
// strided rows and columns each) is the mass of its cells averaged over the
// block's strided rows, X[I, J] = (S / bs) sum P[r, c].  Each block row then
// keeps the smallest descending prefix of X[I, 0..I] (ties: lower J) that
// reaches the threshold of the row's mass, plus its diagonal block.
//
// z is one dense product per head: the strided rows' features are the S
// tokens of the group in order, the strided columns' features the S tokens
// of the key group in reverse order, so z = Q' K'^T with K = S d.  Both are
// views of Q and K through a three-dimensional tensor map (token c S + j is
// element (x, j H + h, c)), so nothing is copied.
//
// Two passes over the causal cells, both tcgen05 products of one 128-row
// strided tile against 256-column super-tiles (M = 128, N = 256, two
// 256-column TMEM accumulators so one super-tile's epilogue runs under the
// next one's products):
//   pass 1: each epilogue thread owns a strided row and keeps its running
//     (max, sum) in the log2 domain;
//   pass 2: each thread forms its row's probabilities, sums them per block
//     column (a register tree over the columns), and the rows of a block are
//     added across lanes (and warps when a block has 64 or 128 rows); one
//     lane writes each block score.
// One CTA per (128-row tile, head), heaviest tiles first; a loader warp
// streams (Q' 64-feature slab, K' 64-feature slab) stages through a
// four-deep ring, one thread issues the MMAs, four warps read TMEM.
// The selection kernel sorts each block row's scores (bitonic, in shared
// memory), sums them as exact 64-bit fixed-point integers in the sorted
// order, and keeps the shortest prefix reaching the threshold.
#include "attn_common.cuh"
#include "ptx.cuh"

namespace vs {
namespace {

constexpr int kXaThreads = 256;  // warp 0 loader, 1 MMA issuer, 2 tensor memory, 4..7 epilogue
constexpr int kXaStages = 4;
constexpr int kXaQBytes = 128 * 128;  // 128 strided rows x 64 features (bf16)
constexpr int kXaKBytes = 256 * 128;  // 256 strided columns x 64 features
constexpr int kXaStage = kXaQBytes + kXaKBytes;
constexpr int kXaBar = kXaStages * kXaStage;
constexpr int kXaNumBars = 2 * kXaStages + 4;  // full[S], empty[S], acc_full[2], acc_free[2]
constexpr int kXaMisc = kXaBar + kXaNumBars * 8;  // tensor memory slot, abort flag
constexpr int kXaRed = kXaMisc + 16;              // pass 2: [2 buffers][4 warps][2 blocks] partial sums
constexpr int kXaSmem = kXaRed + 2 * 4 * 2 * 4;
constexpr float kXaNegInf = -__builtin_huge_valf();

__device__ __forceinline__ float xa_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int D, bool kPass2>
__global__ void __launch_bounds__(kXaThreads, 1)
    xattn_score_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
                       const XaArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kXaBar);
  uint64_t* full = bars;
  uint64_t* empty = full + kXaStages;
  uint64_t* acc_full = empty + kXaStages;
  uint64_t* acc_free = acc_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kXaMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kXaMisc + 4);
  float* red = reinterpret_cast<float*>(sm + kXaRed);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // heaviest row tiles (most causal columns) first
  const int rt = a.nrt - 1 - (int)(blockIdx.x / a.Hq);
  const int h = (int)(blockIdx.x % a.Hq), kvh = h / a.G;
  const int r0 = rt * 128;
  const int ncol = min(a.R, r0 + 128);  // strided columns with a causal cell in this tile
  const int nst = (ncol + 255) / 256;
  constexpr int kHalves = D / 64;
  const int nstep = a.S * kHalves;  // stages per super-tile

  if (threadIdx.x == 0) {
    for (int i = 0; i < kXaStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_free[i], 4);  // one arrival per epilogue warp
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, 512);  // two 256-column accumulators
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  auto wait = [&](uint64_t* bar, uint32_t parity, int where) -> bool {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (mbar_wait(bar, parity, kWaitLimitNs)) return true;
    *abort_flag = 1;
    report_timeout_first(a.status, kTagXattn * 100 + (kPass2 ? 50 : 0) + where);
    return false;
  };
  auto wait_warp = [&](uint64_t* bar, uint32_t parity, int where) -> bool {
    return __all_sync(0xffffffffu, wait(bar, parity, where));
  };

  if (warp == 0) {
    // ------------------------------------------------------------ loader
    if (lane == 0) {
      tma_prefetch_desc(&mQ);
      tma_prefetch_desc(&mK);
      int it = 0;
      bool ok = true;
      for (int st = 0; st < nst && ok; ++st) {
        for (int step = 0; step < nstep; ++step, ++it) {
          const int s = it % kXaStages;
          if (!wait(&empty[s], ((it / kXaStages) & 1) ^ 1, 1)) {
            ok = false;
            break;
          }
          const int j = step / kHalves, hf = step % kHalves;
          uint8_t* base = sm + s * kXaStage;
          mbar_arrive_expect_tx(&full[s], (uint32_t)kXaStage);
          // query token r S + j; key token c S + S-1-j (rows and columns
          // beyond R arrive as zeros and are masked)
          const int yq = j * a.Hq + h, yk = (a.S - 1 - j) * a.Hkv + kvh;
          tma_load_3d(base, &mQ, &full[s], hf * 64, yq, r0);
          tma_load_3d(base + 8192, &mQ, &full[s], hf * 64, yq, r0 + 64);
#pragma unroll
          for (int u = 0; u < 4; ++u)
            tma_load_3d(base + kXaQBytes + u * 8192, &mK, &full[s], hf * 64, yk, st * 256 + 64 * u);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdesc = idesc_bf16(128, 256, false, false);
      int it = 0;
      bool ok = true;
      for (int st = 0; st < nst && ok; ++st) {
        const int acc = st & 1;
        if (st >= 2 && !wait(&acc_free[acc], ((st >> 1) - 1) & 1, 2)) break;
        tc_fence_after();
        const uint32_t tacc = tbase + (uint32_t)(acc * 256);
        for (int step = 0; step < nstep; ++step, ++it) {
          const int s = it % kXaStages;
          if (!wait(&full[s], (it / kXaStages) & 1, 3)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t base = smem_u32(sm + s * kXaStage);
          const uint64_t ad0 = sdesc_sw128(base, 16, 1024);
          const uint64_t bd0 = sdesc_sw128(base + kXaQBytes, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_ss(tacc, sdesc_add(ad0, kk * 32), sdesc_add(bd0, kk * 32), kIdesc, (step > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&empty[s]);
        }
        if (ok) umma_commit(&acc_full[acc]);
      }
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue
    const int q = warp - 4;  // tensor memory lane quadrant
    const int i = q * 32 + lane;
    const int r = r0 + i;  // this thread's strided row
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const float c2 = a.c2;
    // columns c < climit hold this row's causal cells (none for rows past R)
    const int climit = r < a.R ? r + 1 : 0;
    if (!kPass2) {
      float m = kXaNegInf, l = 0.f;
      for (int st = 0; st < nst; ++st) {
        if (!wait_warp(&acc_full[st & 1], (st >> 1) & 1, 4)) break;
        tc_fence_after();
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          uint32_t x[128];
#pragma unroll
          for (int c0 = 0; c0 < 128; c0 += 32)
            tmem_ld32(tbase + (uint32_t)((st & 1) * 256 + half * 128 + c0) + lane_off, x + c0);
          tmem_ld_wait();
          if (half == 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_free[st & 1]);
          }
          const int lim = climit - (st * 256 + half * 128);  // valid columns of this half
          float mx = kXaNegInf;
#pragma unroll
          for (int j = 0; j < 128; ++j) {
            const float v = j < lim ? __uint_as_float(x[j]) * c2 : kXaNegInf;
            x[j] = __float_as_uint(v);
            mx = fmaxf(mx, v);
          }
          const float mn = fmaxf(m, mx);
          if (mn != kXaNegInf) {
            float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
            for (int j = 0; j < 128; j += 4) {
              s0 += xa_exp2(__uint_as_float(x[j]) - mn);
              s1 += xa_exp2(__uint_as_float(x[j + 1]) - mn);
              s2 += xa_exp2(__uint_as_float(x[j + 2]) - mn);
              s3 += xa_exp2(__uint_as_float(x[j + 3]) - mn);
            }
            l = l * xa_exp2(m - mn) + ((s0 + s1) + (s2 + s3));
            m = mn;
          }
        }
      }
      if (r < a.R && !*abort_flag) a.rs[(size_t)h * a.R + r] = make_float2(m, l);
    } else {
      // the row's (max, 1 / sum) from pass 1
      float M = 0.f, inv = 0.f;
      if (r < a.R) {
        const float2 t = a.rs[(size_t)h * a.R + r];
        M = t.x;
        inv = t.y > 0.f ? 1.0f / t.y : 0.f;
      }
      const int bsS = a.bsS;
      int lb = 0;
      while ((1 << lb) < bsS) ++lb;
      float* Xrow = a.X + ((size_t)h * a.nb + (r < a.R ? r >> lb : 0)) * a.nb;
      int rb = 0;
      // Every epilogue warp runs all nst x 2 iterations (a failed wait only
      // skips the work), so the named barrier of the 64- and 128-row blocks
      // always sees all four warps.
      for (int st = 0; st < nst; ++st) {
        const bool ok = wait_warp(&acc_full[st & 1], (st >> 1) & 1, 4);
        if (ok) tc_fence_after();
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          const int c0 = st * 256 + half * 128;
          uint32_t x[128];
          if (ok) {
#pragma unroll
            for (int cc = 0; cc < 128; cc += 32)
              tmem_ld32(tbase + (uint32_t)((st & 1) * 256 + half * 128 + cc) + lane_off, x + cc);
            tmem_ld_wait();
            if (half == 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&acc_free[st & 1]);
            }
            const int lim = climit - c0;
#pragma unroll
            for (int j = 0; j < 128; ++j)
              x[j] = __float_as_uint(j < lim ? xa_exp2(fmaf(__uint_as_float(x[j]), c2, -M)) * inv : 0.f);
            // block-column sums: after level t, x[j] (j a multiple of 2^(t+1))
            // holds the sum of columns j .. j + 2^(t+1) - 1
#pragma unroll
            for (int t = 0; t < 7; ++t)
              if (t < lb) {
#pragma unroll
                for (int j = 0; j < 128; j += 2 << t)
                  x[j] = __float_as_uint(__uint_as_float(x[j]) + __uint_as_float(x[j + (1 << t)]));
              }
          }
          const int jb0 = c0 >> lb;  // block column of this half's first block
          if (bsS <= 32) {
            // a block's rows are bsS consecutive lanes
            if (ok) {
#pragma unroll
              for (int j = 0; j < 128; j += 4)
                if ((j & (bsS - 1)) == 0) {
                  float v = __uint_as_float(x[j]);
                  for (int o = 1; o < bsS; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                  const int J = jb0 + (j >> lb);
                  if ((lane & (bsS - 1)) == 0 && r < a.R && J < a.nb) Xrow[J] = v * a.inv_bsS;
                }
            }
          } else {
            // 64 rows (two warps) or 128 rows (four warps) per block: warp
            // sums through shared memory, added in warp order by warp 4
            float v0 = ok ? __uint_as_float(x[0]) : 0.f, v1 = ok ? __uint_as_float(x[64]) : 0.f;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
              v0 += __shfl_xor_sync(0xffffffffu, v0, o);
              v1 += __shfl_xor_sync(0xffffffffu, v1, o);
            }
            float* rbuf = red + rb * 8;
            if (lane == 0) {
              rbuf[q * 2] = v0;
              rbuf[q * 2 + 1] = v1;
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
            if (ok && q == 0) {
              if (bsS == 64 && lane < 4) {
                const int br = lane >> 1, bc = lane & 1;  // block row in the tile, block column in the half
                const float v = rbuf[(2 * br) * 2 + bc] + rbuf[(2 * br + 1) * 2 + bc];
                const int Ib = (r0 >> 6) + br, Jb = jb0 + bc;
                if (Ib * 64 < a.R && Jb < a.nb) a.X[((size_t)h * a.nb + Ib) * a.nb + Jb] = v * a.inv_bsS;
              } else if (bsS == 128 && lane == 0) {
                const float v = ((rbuf[0] + rbuf[2]) + rbuf[4]) + rbuf[6];
                const int Ib = r0 >> 7, Jb = jb0;
                if (Ib * 128 < a.R && Jb < a.nb) a.X[((size_t)h * a.nb + Ib) * a.nb + Jb] = v * a.inv_bsS;
              }
            }
            rb ^= 1;
          }
        }
      }
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tbase, 512);
}

// Block-wide sum and exclusive scan of 64-bit integers (256 threads).
__device__ unsigned long long xa_block_sum(unsigned long long v, unsigned long long* wbuf) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) wbuf[warp] = v;
  __syncthreads();
  unsigned long long t = 0;
  for (int w = 0; w < kXaThreads / 32; ++w) t += wbuf[w];
  return t;
}
__device__ unsigned long long xa_block_exscan(unsigned long long v, unsigned long long* wbuf) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned long long inc = v;
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  __syncthreads();
  if (lane == 31) wbuf[warp] = inc;
  __syncthreads();
  unsigned long long before = 0;
  for (int w = 0; w < warp; ++w) before += wbuf[w];
  return before + inc - v;
}

// One CTA per (block row I, head h): the kept block columns of row I.
// Sort keys: (score bits << 32) | (2^32 - 1 - J), sorted descending, so equal
// scores come lower J first; scores are non-negative fp32, whose bit
// patterns order like the values.
__global__ void __launch_bounds__(kXaThreads) xattn_select_kernel(const XaArgs a) {
  extern __shared__ unsigned long long xa_keys[];
  __shared__ unsigned long long wbuf[kXaThreads / 32];
  __shared__ uint32_t words[512];
  __shared__ int kfirst;
  const int I = blockIdx.x, h = blockIdx.y;
  const int n = I + 1;
  int npad = 1;
  while (npad < n) npad <<= 1;
  const float* row = a.X + ((size_t)h * a.nb + I) * a.nb;
  for (int j = threadIdx.x; j < npad; j += kXaThreads)
    xa_keys[j] = j < n ? ((unsigned long long)__float_as_uint(row[j]) << 32) | (unsigned long long)(0xffffffffu - (uint32_t)j)
                       : 0ull;
  for (int w = threadIdx.x; w < a.nw; w += kXaThreads) words[w] = 0u;
  if (threadIdx.x == 0) kfirst = n;
  __syncthreads();
  // bitonic sort, descending
  for (int k = 2; k <= npad; k <<= 1)
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < npad; i += kXaThreads) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const unsigned long long u = xa_keys[i], v = xa_keys[ixj];
          if ((i & k) == 0 ? (u < v) : (u > v)) {
            xa_keys[i] = v;
            xa_keys[ixj] = u;
          }
        }
      }
      __syncthreads();
    }
  // scores as exact fixed-point integers: x * 2^60, truncated (a block row's
  // scores sum to about 1, so every partial sum stays below 2^62)
  auto quant = [](unsigned long long key) -> unsigned long long {
    return (unsigned long long)__float2ull_rz(ldexpf(__uint_as_float((uint32_t)(key >> 32)), 60));
  };
  // each thread owns a run of consecutive sorted positions
  const int seg = (npad + kXaThreads - 1) / kXaThreads;
  const int b0 = (int)threadIdx.x * seg, b1 = min(b0 + seg, n);
  unsigned long long mine = 0, npos = 0;
  for (int p = b0; p < b1; ++p) {
    mine += quant(xa_keys[p]);
    npos += (xa_keys[p] >> 32) != 0ull;
  }
  int kc;
  if (a.threshold >= 1.f) {
    kc = (int)xa_block_sum(npos, wbuf);  // every positive score (they sort first)
  } else {
    const unsigned long long tot = xa_block_sum(mine, wbuf);
    unsigned long long target = (unsigned long long)((double)a.threshold * (double)tot);
    if ((double)target < (double)a.threshold * (double)tot) ++target;
    if (target < 1) target = 1;
    unsigned long long run = xa_block_exscan(mine, wbuf);
    for (int p = b0; p < b1; ++p) {
      run += quant(xa_keys[p]);
      if (run >= target) {
        atomicMin(&kfirst, p + 1);
        break;
      }
    }
    __syncthreads();
    kc = kfirst;
  }
  for (int p = threadIdx.x; p < kc; p += kXaThreads) {
    const uint32_t J = 0xffffffffu - (uint32_t)xa_keys[p];
    atomicOr(&words[J >> 5], 1u << (J & 31));
  }
  if (threadIdx.x == 0) atomicOr(&words[I >> 5], 1u << (I & 31));  // the diagonal block
  __syncthreads();
  uint32_t* out = a.mask + ((size_t)h * a.nb + I) * a.nw;
  int c = 0;
  for (int w = threadIdx.x; w < a.nw; w += kXaThreads) {
    out[w] = words[w];
    c += __popc(words[w]);
  }
  const int cnt = (int)xa_block_sum((unsigned long long)c, wbuf);
  if (threadIdx.x == 0) {
    a.cnt[(size_t)h * a.nb + I] = cnt;
    const unsigned long long bs = (unsigned long long)a.bs;
    atomicAdd(&a.active[h], (unsigned long long)(cnt - 1) * bs * bs + bs * (bs + 1) / 2);
  }
}

template <int D>
cudaError_t launch_scores(const XaArgs& a, cudaStream_t s) {
  CUtensorMap mQ, mK;
  if (!make_map_strided(&mQ, a.Q, a.R, a.Hq, D, a.S) || !make_map_strided(&mK, a.K, a.R, a.Hkv, D, a.S))
    return cudaErrorInvalidValue;
  const size_t smem = kXaSmem + 1024;
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(xattn_score_kernel<D, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)smem)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(xattn_score_kernel<D, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)smem)) != cudaSuccess)
    return e;
  const int grid = a.nrt * a.Hq;
  xattn_score_kernel<D, false><<<grid, kXaThreads, smem, s>>>(mQ, mK, a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  xattn_score_kernel<D, true><<<grid, kXaThreads, smem, s>>>(mQ, mK, a);
  return cudaGetLastError();
}

}  // namespace

size_t xattn_select_smem(int nb) {
  size_t npad = 1;
  while (npad < (size_t)nb) npad <<= 1;
  return npad * sizeof(unsigned long long);
}

cudaError_t launch_xattn(const XaArgs& a, cudaStream_t s) {
  cudaError_t e;
  // block scores above the diagonal stay zero; the kept-entry counts are sums
  if ((e = cudaMemsetAsync(a.X, 0, (size_t)a.Hq * a.nb * a.nb * sizeof(float), s)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(a.active, 0, (size_t)a.Hq * sizeof(unsigned long long), s)) != cudaSuccess) return e;
  if ((e = (a.d == 128 ? launch_scores<128>(a, s) : launch_scores<64>(a, s))) != cudaSuccess) return e;
  const size_t smem = xattn_select_smem(a.nb);
  if ((e = cudaFuncSetAttribute(xattn_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
      cudaSuccess)
    return e;
  xattn_select_kernel<<<dim3(a.nb, a.Hq), kXaThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace vs
