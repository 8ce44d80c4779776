// Sparse-index scoring on the tensor cores (last_q = 64).
//
// MTraining review, section "分布式稀疏索引近似": the last last_q query rows
// are scored against every key, p = softmax over the causal keys per row,
// and the attention mass is summed along verticals (v[m] = sum over rows of
// p) and slash bands (S[B] = sum of p over the entries of band B).  With
// last_q = 64 every index row lies in the last 64-token block, hence in the
// last band row of any stripe width, so a band's mass is the vertical mass
// of its keys: S[B] = sum of v[m] over the keys m of band B.
//
// Two passes over K, both tcgen05 products of a pair of query heads (128
// rows: two heads x 64 rows, one head and zeros when the group has an odd
// head left) with 128-key tiles:
//   pass 1, rows on M: S = Q K^T; each epilogue thread owns one row and half
//     of the keys and keeps their running (max, sum) in the log2 domain,
//     written per key chunk and half;
//   pass 2, keys on M: S^T = K Q^T; each epilogue thread owns one key and one
//     head of the pair, forms p for the head's 64 rows from the rows' (max,
//     1 / sum) combined over the partials, and sums them into v; the 64-key
//     block sums of v go to a small table that the slash kernel adds up per
//     band.
// One CTA per (key chunk, head pair, key/value head); a loader warp stages
// the pair's Q rows once and streams K tiles through a three-deep ring, one
// thread issues the MMAs into two TMEM accumulators, eight warps read them
// (two per lane quadrant, each 64 of the tile's 128 columns).
#include "attn_common.cuh"
#include "ptx.cuh"

namespace vs {
namespace {

constexpr int kIxThreads = 384;  // warp 0 loader, 1 MMA issuer, 2 tensor memory, 4..11 epilogue
constexpr int kIxStages = 3;
constexpr float kIxNegInf = -__builtin_huge_valf();

template <int D>
struct IxLayout {
  static constexpr int kHalf = 128 * 128;            // 128 rows x one 64-wide d half (bf16)
  static constexpr int kTile = (D / 64) * kHalf;     // 128 rows (or keys) x D
  static constexpr int kQ = 0;                       // the head pair's query rows (stationary)
  static constexpr int kK = kTile;                   // key tile ring
  static constexpr int kBar = kK + kIxStages * kTile;
  // q_full, k_full[S], k_empty[S], acc_full[2], acc_free[2]
  static constexpr int kNumBars = 1 + 2 * kIxStages + 4;
  static constexpr int kMisc = kBar + kNumBars * 8;  // tensor memory slot, abort flag
  static constexpr int kRow = kMisc + 16;            // pass 2: (max, 1 / sum) of the 128 rows
  static constexpr int kRed = kRow + 128 * 8;        // pass 2: per-warp block sums [2 buffers][2 heads][4]
  static constexpr int kHist = kRed + 2 * 4 * 2 * 4;  // pass 2: [2 heads][2048] counts of v by key >> 20
  static constexpr int kSmem = kHist + 2 * 2048 * 4;
};

__device__ __forceinline__ float ix_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace

IxTcGrid index_tc_grid(int L, int Hq, int Hkv) {
  IxTcGrid c;
  const int G = Hq / Hkv;
  c.npairs = (G + 1) / 2;
  const int ntiles = (L + 127) / 128;
  int C = 148 / (c.npairs * Hkv);
  if (C < 1) C = 1;
  if (C > ntiles) C = ntiles;
  c.tpc = (ntiles + C - 1) / C;
  c.C = (ntiles + c.tpc - 1) / c.tpc;
  return c;
}

namespace {

template <int D, bool kPass2>
__global__ void __launch_bounds__(kIxThreads, 1)
    index_tc_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
                    const IndexArgs a, const IxTcGrid c) {
  using Ly = IxLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Ly::kBar);
  uint64_t* q_full = bars;
  uint64_t* k_full = q_full + 1;
  uint64_t* k_empty = k_full + kIxStages;
  uint64_t* acc_full = k_empty + kIxStages;
  uint64_t* acc_free = acc_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + Ly::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + Ly::kMisc + 4);
  float2* rowst = reinterpret_cast<float2*>(sm + Ly::kRow);
  float* red = reinterpret_cast<float*>(sm + Ly::kRed);  // [2 buffers][2 heads][4 warps]
  uint32_t* hist = reinterpret_cast<uint32_t*>(sm + Ly::kHist);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = blockIdx.x, pair = blockIdx.y, g = blockIdx.z;
  const int ha = g * a.G + 2 * pair;
  const bool has_b = 2 * pair + 1 < a.G;
  const int hb = has_b ? ha + 1 : ha;
  const int ntiles = (a.L + 127) / 128;
  const int t0 = chunk * c.tpc;
  const int nt = max(0, min(ntiles, t0 + c.tpc) - t0);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < kIxStages; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_free[i], 8);  // one arrival per epilogue warp
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, 256);  // two 128-column accumulators
    tmem_relinquish();
  }
  if (kPass2)
    for (int j = threadIdx.x; j < 2 * 2048; j += kIxThreads) hist[j] = 0u;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  auto wait = [&](uint64_t* bar, uint32_t parity, int where) -> bool {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (mbar_wait(bar, parity, kWaitLimitNs)) return true;
    *abort_flag = 1;
    report_timeout_first(a.status, kTagIndex * 100 + (kPass2 ? 50 : 0) + where);
    return false;
  };
  auto wait_warp = [&](uint64_t* bar, uint32_t parity, int where) -> bool {
    return __all_sync(0xffffffffu, wait(bar, parity, where));
  };

  if (warp == 0) {
    // ------------------------------------------------------------ loader
    // the pair's query rows once (zeros for a missing second head), then
    // the chunk's key tiles
    if (!has_b) {
      for (int hf = 0; hf < D / 64; ++hf) {
        uint4* z = reinterpret_cast<uint4*>(sm + Ly::kQ + hf * Ly::kHalf + 8192);
#pragma unroll
        for (int k = 0; k < 16; ++k) z[k * 32 + lane] = make_uint4(0u, 0u, 0u, 0u);
      }
      fence_proxy_async_smem();
    }
    __syncwarp();
    if (lane == 0) {
      tma_prefetch_desc(&mQ);
      tma_prefetch_desc(&mK);
      mbar_arrive_expect_tx(q_full, (uint32_t)((has_b ? 2 : 1) * (D / 64) * 8192));
      for (int hf = 0; hf < D / 64; ++hf) {
        tma_load_3d(sm + Ly::kQ + hf * Ly::kHalf, &mQ, q_full, hf * 64, ha, a.L - 64);
        if (has_b) tma_load_3d(sm + Ly::kQ + hf * Ly::kHalf + 8192, &mQ, q_full, hf * 64, hb, a.L - 64);
      }
      for (int t = 0; t < nt; ++t) {
        const int s = t % kIxStages;
        if (!wait(&k_empty[s], ((t / kIxStages) & 1) ^ 1, 1)) break;
        uint8_t* kt = sm + Ly::kK + s * Ly::kTile;
        mbar_arrive_expect_tx(&k_full[s], (uint32_t)Ly::kTile);
        // keys beyond L arrive as zeros (the box reads out of bounds) and are masked
        for (int hf = 0; hf < D / 64; ++hf)
          for (int j = 0; j < 2; ++j)
            tma_load_3d(kt + hf * Ly::kHalf + j * 8192, &mK, &k_full[s], hf * 64, g, (t0 + t) * 128 + 64 * j);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdesc = idesc_bf16(128, 128, false, false);
      const uint32_t qa = smem_u32(sm + Ly::kQ);
      if (wait(q_full, 0, 2)) {
        for (int t = 0; t < nt; ++t) {
          const int s = t % kIxStages;
          if (!wait(&k_full[s], (t / kIxStages) & 1, 3)) break;
          if (t >= 2 && !wait(&acc_free[t & 1], ((t >> 1) - 1) & 1, 4)) break;
          tc_fence_after();
          const uint32_t ka = smem_u32(sm + Ly::kK + s * Ly::kTile);
          // pass 1: rows x keys = Q K^T; pass 2: keys x rows = K Q^T
          const uint64_t ad0 = sdesc_sw128(kPass2 ? ka : qa, 16, 1024);
          const uint64_t bd0 = sdesc_sw128(kPass2 ? qa : ka, 16, 1024);
          const uint32_t tacc = tbase + (uint32_t)((t & 1) * 128);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * Ly::kHalf + (kk & 3) * 32;
            umma_ss(tacc, sdesc_add(ad0, off), sdesc_add(bd0, off), kIdesc, kk > 0 ? 1u : 0u);
          }
          umma_commit(&k_empty[s]);
          umma_commit(&acc_full[t & 1]);
        }
      }
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue
    // two warps per tensor memory lane quadrant, each reading half of the
    // tile's 128 columns: pass 1 keys 64 hc .. 64 hc + 63, pass 2 the rows
    // of one head of the pair (hc = 0: head a, 1: head b)
    const int q = (warp - 4) & 3;  // lane quadrant
    const int hc = (warp - 4) >> 2;
    const int i = q * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const float c2 = a.scale_log2;
    const int nq = a.L - 64;  // token of the first index row
    if (!kPass2) {
      // thread = row i of the pair: running max / sum over this chunk's keys
      // in its column half, written as one of the chunk's two partials
      const int n = nq + (i & 63);
      float m = kIxNegInf, l = 0.f;
      for (int t = 0; t < nt; ++t) {
        if (!wait_warp(&acc_full[t & 1], (t >> 1) & 1, 5)) break;
        tc_fence_after();
        uint32_t x[64];
        const uint32_t ta = tbase + (uint32_t)((t & 1) * 128 + 64 * hc) + lane_off;
        tmem_ld32(ta, x);
        tmem_ld32(ta + 32, x + 32);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_free[t & 1]);
        const int k0 = (t0 + t) * 128 + 64 * hc;
        const bool masked = k0 + 63 > nq;  // the half reaches the index rows' own block
        float mx = kIxNegInf;
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          float v = __uint_as_float(x[j]) * c2;
          if (masked && k0 + j > n) v = kIxNegInf;
          x[j] = __float_as_uint(v);
          mx = fmaxf(mx, v);
        }
        const float mn = fmaxf(m, mx);
        if (mn != kIxNegInf) {
          float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
          for (int j = 0; j < 64; j += 4) {
            s0 += ix_exp2(__uint_as_float(x[j]) - mn);
            s1 += ix_exp2(__uint_as_float(x[j + 1]) - mn);
            s2 += ix_exp2(__uint_as_float(x[j + 2]) - mn);
            s3 += ix_exp2(__uint_as_float(x[j + 3]) - mn);
          }
          l = l * ix_exp2(m - mn) + ((s0 + s1) + (s2 + s3));
          m = mn;
        }
      }
      const bool valid = i < 64 || has_b;
      if (valid) {
        const int h = i < 64 ? ha : hb;
        a.part[(size_t)(2 * chunk + hc) * a.Hq * 64 + (size_t)h * 64 + (i & 63)] = make_float2(m, l);
      }
    } else {
      // the pair's 128 rows: (max, 1 / sum) combined over the pass-1
      // partials (two per key chunk)
      if (hc == 0) {
        const bool valid = i < 64 || has_b;
        const size_t prow = (size_t)(i < 64 ? ha : hb) * 64 + (i & 63);
        float M = kIxNegInf, l = 0.f;
        if (valid) {
          for (int ch = 0; ch < 2 * c.C; ++ch) M = fmaxf(M, a.part[(size_t)ch * a.Hq * 64 + prow].x);
          for (int ch = 0; ch < 2 * c.C; ++ch) {
            const float2 pt = a.part[(size_t)ch * a.Hq * 64 + prow];
            if (pt.x != kIxNegInf) l += pt.y * ix_exp2(pt.x - M);
          }
        }
        rowst[i] = (valid && l > 0.f) ? make_float2(M, 1.0f / l) : make_float2(0.f, 0.f);
      }
      asm volatile("bar.sync 1, 256;" ::: "memory");
      // thread = key i of the tile: p over this warp's head's 64 rows.  Every
      // warp runs all nt iterations (a failed wait only skips the work), so
      // the per-head named barrier always sees the head's four warps.
      const bool head_on = hc == 0 || has_b;
      const int h = hc ? hb : ha;
      const float2* rs = rowst + 64 * hc;
      for (int t = 0; t < nt; ++t) {
        const bool ok = wait_warp(&acc_full[t & 1], (t >> 1) & 1, 5);
        const int k0 = (t0 + t) * 128;
        const int k = k0 + i;
        float va = 0.f;
        if (ok) {
          tc_fence_after();
          uint32_t x[64];
          const uint32_t ta = tbase + (uint32_t)((t & 1) * 128 + 64 * hc) + lane_off;
          tmem_ld32(ta, x);
          tmem_ld32(ta + 32, x + 32);
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_free[t & 1]);
          const bool masked = k0 + 127 > nq;
          float v0 = 0.f, v1 = 0.f, v2 = 0.f, v3 = 0.f;
#pragma unroll
          for (int cc = 0; cc < 64; cc += 4) {
            float p0 = ix_exp2(fmaf(__uint_as_float(x[cc]), c2, -rs[cc].x)) * rs[cc].y;
            float p1 = ix_exp2(fmaf(__uint_as_float(x[cc + 1]), c2, -rs[cc + 1].x)) * rs[cc + 1].y;
            float p2 = ix_exp2(fmaf(__uint_as_float(x[cc + 2]), c2, -rs[cc + 2].x)) * rs[cc + 2].y;
            float p3 = ix_exp2(fmaf(__uint_as_float(x[cc + 3]), c2, -rs[cc + 3].x)) * rs[cc + 3].y;
            if (masked) {
              // causal: row cc of the head is token nq + cc
              if (k > nq + cc) p0 = 0.f;
              if (k > nq + cc + 1) p1 = 0.f;
              if (k > nq + cc + 2) p2 = 0.f;
              if (k > nq + cc + 3) p3 = 0.f;
            }
            v0 += p0;
            v1 += p1;
            v2 += p2;
            v3 += p3;
          }
          va = (v0 + v1) + (v2 + v3);
          if (k < a.L && head_on) {
            a.v[(size_t)h * a.L + k] = va;
            atomicAdd(&hist[hc * 2048 + min(__float_as_uint(va) >> 20, 2047u)], 1u);
          }
        }
        // 64-key block sums (keys beyond L hold zeros): warps of quadrants
        // 0-1 hold the tile's first block, 2-3 its second
        float wa = va;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) wa += __shfl_xor_sync(0xffffffffu, wa, o);
        float* rb = red + (t & 1) * 8 + hc * 4;
        if (lane == 0) rb[q] = wa;
        asm volatile("bar.sync %0, 128;" ::"r"(2 + hc) : "memory");
        if (ok && head_on && q == 0 && lane < 2) {
          const int blk = k0 / 64 + lane;
          if (blk < a.ntile) a.T64[(size_t)h * a.ntile + blk] = rb[2 * lane] + rb[2 * lane + 1];
        }
      }
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tbase, 256);
  if (kPass2 && !*abort_flag)
    // this CTA's counts into the heads' histograms (non-zero bins only)
    for (int j = threadIdx.x; j < (has_b ? 2 : 1) * 2048; j += kIxThreads) {
      const uint32_t cnt = hist[j];
      if (cnt) atomicAdd(&a.vhist[(size_t)(j < 2048 ? ha : hb) * 2048 + (j & 2047)], cnt);
    }
}

// S[h][B] = sum of the 64-key block masses of band B: key blocks
// (J - B) W .. (J - B) W + W - 1, J = nbs - 1 the index rows' band row.
__global__ void index_tc_slash_kernel(const IndexArgs a) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= a.Hq * a.nbs) return;
  const int h = idx / a.nbs, B = idx % a.nbs;
  const int W = a.bs / 64;
  const float* T = a.T64 + (size_t)h * a.ntile + (size_t)(a.nbs - 1 - B) * W;
  float s = 0.f;
  for (int w = 0; w < W; ++w) s += T[w];
  a.S[idx] = s;
}

template <int D>
cudaError_t launch_tc(const IndexArgs& a, cudaStream_t s) {
  using Ly = IxLayout<D>;
  CUtensorMap mQ, mK;
  if (!make_map_heads(&mQ, a.Q, a.L, a.Hq, D) || !make_map_heads(&mK, a.K, a.L, a.Hkv, D))
    return cudaErrorInvalidValue;
  const IxTcGrid c = index_tc_grid(a.L, a.Hq, a.Hkv);
  const size_t smem = Ly::kSmem + 1024;
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(index_tc_kernel<D, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)smem)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(index_tc_kernel<D, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)smem)) != cudaSuccess)
    return e;
  const dim3 grid(c.C, c.npairs, a.Hkv);
  if ((e = cudaMemsetAsync(a.vhist, 0, (size_t)a.Hq * 2048 * sizeof(uint32_t), s)) != cudaSuccess) return e;
  index_tc_kernel<D, false><<<grid, kIxThreads, smem, s>>>(mQ, mK, a, c);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  index_tc_kernel<D, true><<<grid, kIxThreads, smem, s>>>(mQ, mK, a, c);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int n = a.Hq * a.nbs;
  index_tc_slash_kernel<<<(n + 255) / 256, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

bool index_tc_supported(const IndexArgs& a) { return a.last_q == 64 && (a.d == 64 || a.d == 128) && a.L >= 64; }

cudaError_t launch_index_scores_tc(const IndexArgs& a, cudaStream_t s) {
  return a.d == 128 ? launch_tc<128>(a, s) : launch_tc<64>(a, s);
}

}  // namespace vs
