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
// The selection kernel gives each block row one warp, which finds the
// row's threshold score by a radix descent over exact 64-bit fixed-point
// sums (no sort) and keeps the scores above it, then ties in index order,
// up to the threshold's share.
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
__device__ __forceinline__ float xa_log2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// kBsS: strided rows per block (pass 2 only; 0 in pass 1)
template <int D, bool kPass2, int kBsS>
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
    if constexpr (!kPass2) {
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
      // the row's log2 normaliser from pass 1: p = exp2(z c2 - (max + log2 sum))
      float Mn = 0.f;
      if (r < a.R) {
        const float2 t = a.rs[(size_t)h * a.R + r];
        Mn = t.x + xa_log2(t.y);
      }
      constexpr int kLb = kBsS <= 4 ? 2 : kBsS <= 8 ? 3 : kBsS <= 16 ? 4 : kBsS <= 32 ? 5 : kBsS <= 64 ? 6 : 7;
      constexpr int kNb = 128 / kBsS;  // block columns per 128-column half
      float* Xrow = a.X + ((size_t)h * a.nb + (r < a.R ? r >> kLb : 0)) * a.nb;
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
          float v[kNb];
          if (ok) {
            uint32_t x[128];
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
            if (__all_sync(0xffffffffu, lim >= 128)) {
#pragma unroll
              for (int j = 0; j < 128; ++j) x[j] = __float_as_uint(xa_exp2(fmaf(__uint_as_float(x[j]), c2, -Mn)));
            } else {
#pragma unroll
              for (int j = 0; j < 128; ++j)
                x[j] = __float_as_uint(j < lim ? xa_exp2(fmaf(__uint_as_float(x[j]), c2, -Mn)) : 0.f);
            }
            // block-column sums: after level t, x[j] (j a multiple of 2^(t+1))
            // holds the sum of columns j .. j + 2^(t+1) - 1
#pragma unroll
            for (int t = 0; t < kLb; ++t)
#pragma unroll
              for (int j = 0; j < 128; j += 2 << t)
                x[j] = __float_as_uint(__uint_as_float(x[j]) + __uint_as_float(x[j + (1 << t)]));
#pragma unroll
            for (int b = 0; b < kNb; ++b) v[b] = __uint_as_float(x[b * kBsS]);
          }
          const int jb0 = c0 >> kLb;  // block column of this half's first block
          if constexpr (kBsS <= 32) {
            // a block's rows are kBsS consecutive lanes: reduce-scatter the
            // kNb block sums across them, halving the list per exchange
            if (ok) {
              int base = 0;  // first block column held by this lane
              constexpr int kSteps = kLb < (kNb > 1 ? __builtin_ctz(kNb) : 0) ? kLb : (kNb > 1 ? __builtin_ctz(kNb) : 0);
#pragma unroll
              for (int sstep = 0; sstep < kSteps; ++sstep) {
                const int o = kBsS >> (sstep + 1);
                const int cnt = kNb >> sstep, hlf = cnt >> 1;
                const bool upper = (lane & o) != 0;
#pragma unroll
                for (int i = 0; i < hlf; ++i) {
                  const float send = upper ? v[i] : v[i + hlf];
                  const float keep = upper ? v[i + hlf] : v[i];
                  v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                }
                if (upper) base += hlf;
              }
              constexpr int kLeft = kNb >> kSteps;  // block sums held per lane
              // lanes still sharing those blocks: the lower offsets not used
              constexpr int kRest = kBsS >> kSteps;
#pragma unroll
              for (int o = kRest >> 1; o > 0; o >>= 1)
#pragma unroll
                for (int i = 0; i < kLeft; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i], o);
              if ((lane & (kRest - 1)) == 0 && r < a.R) {
#pragma unroll
                for (int i = 0; i < kLeft; ++i)
                  if (jb0 + base + i < a.nb) Xrow[jb0 + base + i] = v[i] * a.inv_bsS;
              }
            }
          } else {
            // 64 rows (two warps) or 128 rows (four warps) per block: warp
            // sums through shared memory, added in warp order by warp 4
            float v0 = ok ? v[0] : 0.f, v1 = (ok && kNb > 1) ? v[kNb > 1 ? 1 : 0] : 0.f;
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
              if (kBsS == 64 && lane < 4) {
                const int br = lane >> 1, bc = lane & 1;  // block row in the tile, block column in the half
                const float sum = rbuf[(2 * br) * 2 + bc] + rbuf[(2 * br + 1) * 2 + bc];
                const int Ib = (r0 >> 6) + br, Jb = jb0 + bc;
                if (Ib * 64 < a.R && Jb < a.nb) a.X[((size_t)h * a.nb + Ib) * a.nb + Jb] = sum * a.inv_bsS;
              } else if (kBsS == 128 && lane == 0) {
                const float sum = ((rbuf[0] + rbuf[2]) + rbuf[4]) + rbuf[6];
                const int Ib = r0 >> 7, Jb = jb0;
                if (Ib * 128 < a.R && Jb < a.nb) a.X[((size_t)h * a.nb + Ib) * a.nb + Jb] = sum * a.inv_bsS;
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

// A score as an exact fixed-point integer: x * 2^60, truncated (a block
// row's scores sum to about 1, so every partial sum stays below 2^62).
__device__ __forceinline__ unsigned long long xa_quant(uint32_t key) {
  return (unsigned long long)__float2ull_rz(ldexpf(__uint_as_float(key), 60));
}

__device__ __forceinline__ unsigned long long xa_warp_sum(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

constexpr int kSelWarps = kXaThreads / 32;  // block rows per CTA, one per warp

// Per-warp histogram of one radix level (8-bit digits).
struct XaWarpHist {
  unsigned long long sum[256];
  uint32_t cnt[256];
  uint32_t key[256];  // a key that fell into the bin (exact when the bin holds one)
};

// One warp per (block row I, head h): the kept block columns of row I.
// Scores are non-negative fp32, so their bit patterns order like the
// values.  A most-significant-digit-first radix descent (four 8-bit digits)
// over per-warp histograms of counts and fixed-point sums finds the
// threshold key t: the scores above t sum to less than the target and those
// at or above it reach it.  All scores above t are kept, then the scores
// equal to t in index order until the target is reached (the lower block
// column first among equal scores, as in a stable descending sort).  The
// row is read from global memory (L2) at every level; no block barriers.
__global__ void __launch_bounds__(kXaThreads) xattn_select_kernel(const XaArgs a) {
  __shared__ XaWarpHist hist[kSelWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int I = blockIdx.x * kSelWarps + warp, h = blockIdx.y;
  if (I >= a.nb) return;
  XaWarpHist& H = hist[warp];
  const int n = I + 1;
  const uint32_t* row = reinterpret_cast<const uint32_t*>(a.X) + ((size_t)h * a.nb + I) * a.nb;
  unsigned long long mine = 0;
#pragma unroll 4
  for (int j = lane; j < n; j += 32) mine += xa_quant(__ldg(row + j));
  const unsigned long long tot = xa_warp_sum(mine);
  uint32_t t = 0u;     // threshold key: keep key > t, and ties == t as below
  bool all_ties = false;
  uint32_t ntie = 0u;  // ties kept in index order when not all_ties
  const bool sel = a.threshold < 1.f && tot > 0;  // else every block of positive score
  if (sel) {
    unsigned long long target = (unsigned long long)((double)a.threshold * (double)tot);
    if ((double)target < (double)a.threshold * (double)tot) ++target;
    if (target < 1) target = 1;
    unsigned long long need = target;  // mass still to reach within the current prefix
    uint32_t prefix = 0u, cnt_eq = 0u;
    int lev = 0;
#pragma unroll 1
    for (; lev < 4; ++lev) {
      const int shift = 24 - 8 * lev;
#pragma unroll
      for (int b = lane; b < 256; b += 32) {
        H.sum[b] = 0ull;
        H.cnt[b] = 0u;
      }
      __syncwarp();
      for (int j00 = 0; j00 < n; j00 += 128) {
        // four loads in flight, then the four groups of 32
        uint32_t kb[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) kb[u] = j00 + 32 * u + lane < n ? __ldg(row + j00 + 32 * u + lane) : 0u;
#pragma unroll 1
        for (int u = 0; u < 4; ++u) {
          const int j = j00 + 32 * u + lane;
          const uint32_t k = kb[u];
          const bool in = j < n && (uint32_t)((unsigned long long)k >> (shift + 8)) == prefix;
          // below the first level most groups hold no score of the prefix
          if (__ballot_sync(0xffffffffu, in) == 0u) continue;
          const int d = in ? (int)((k >> shift) & 255u) : -1;
          const unsigned long long q = in ? xa_quant(k) : 0ull;
          // scores of a row often share their leading bits: at most four
          // digits in this group of 32 are reduced across the warp and added
          // once each (a loop every lane runs), more are added one by one
          const unsigned same = __match_any_sync(0xffffffffu, d);
          const unsigned leaders = __ballot_sync(0xffffffffu, in && (__ffs(same) - 1) == lane);
          if (__popc(leaders) > 4) {
            if (in) {
              atomicAdd(&H.sum[d], q);
              atomicAdd(&H.cnt[d], 1u);
              H.key[d] = k;
            }
          } else {
            for (unsigned rest = leaders; rest; rest &= rest - 1) {
              const int src = __ffs(rest) - 1;
              const int dl = __shfl_sync(0xffffffffu, d, src);
              const unsigned long long v = xa_warp_sum((in && d == dl) ? q : 0ull);
              if (lane == src) {
                atomicAdd(&H.sum[dl], v);
                atomicAdd(&H.cnt[dl], (uint32_t)__popc(same));
                H.key[dl] = k;
              }
            }
          }
          __syncwarp();
        }
      }
      // lane u owns bins [8u, 8u + 8); the mass above its range comes from
      // a suffix scan over the lanes; the lane holding the crossing finds
      // the digit d with S(d + 1) < need <= S(d), S the suffix sum
      unsigned long long own = 0;
#pragma unroll
      for (int b = 0; b < 8; ++b) own += H.sum[8 * lane + b];
      unsigned long long inc = own;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_down_sync(0xffffffffu, inc, o);
        if (lane + o < 32) inc += y;
      }
      const unsigned long long above = inc - own;
      const bool mine_x = above < need && above + own >= need;
      uint32_t dg = 0u, ce = 0u, kk = 0u;
      unsigned long long nd = 0ull;
      if (mine_x) {
        unsigned long long acc = above;
        for (int b = 8 * lane + 7; b >= 8 * lane; --b) {
          if (acc + H.sum[b] >= need) {
            dg = (uint32_t)b;
            nd = need - acc;
            ce = H.cnt[b];
            kk = H.key[b];
            break;
          }
          acc += H.sum[b];
        }
      }
      const int src = __ffs(__ballot_sync(0xffffffffu, mine_x)) - 1;
      dg = __shfl_sync(0xffffffffu, dg, src);
      nd = __shfl_sync(0xffffffffu, nd, src);
      ce = __shfl_sync(0xffffffffu, ce, src);
      kk = __shfl_sync(0xffffffffu, kk, src);
      __syncwarp();
      prefix = (prefix << 8) | dg;
      need = nd;
      cnt_eq = ce;
      if (ce == 1u) {
        // one score in the bin: it is the threshold key
        t = kk;
        break;
      }
    }
    if (lev == 4) t = prefix;
    const unsigned long long qt = xa_quant(t);
    unsigned long long k = qt ? (need + qt - 1) / qt : 1;
    if (k < 1) k = 1;
    if (k > cnt_eq) k = cnt_eq;
    ntie = (uint32_t)k;
    all_ties = ntie == cnt_eq;
  }
  // mask words from ballots over the row in index order (word w covers
  // block columns 32 w .. 32 w + 31); ties beyond the first ntie dropped
  uint32_t* out = a.mask + ((size_t)h * a.nb + I) * a.nw;
  uint32_t run = 0, c = 0;
  const bool rank_ties = sel && !all_ties;
#pragma unroll 4
  for (int w = 0; w < a.nw; ++w) {
    const int j = w * 32 + lane;
    const uint32_t k = j < n ? __ldg(row + j) : 0u;
    bool keep = j < n && (k > t || j == I || (sel && all_ties && k == t));
    if (rank_ties) {
      const bool tie = j < n && k == t;
      const unsigned bt = __ballot_sync(0xffffffffu, tie);
      if (tie && run + (uint32_t)__popc(bt & ((1u << lane) - 1u)) < ntie) keep = true;
      run += (uint32_t)__popc(bt);
    }
    const uint32_t word = __ballot_sync(0xffffffffu, keep);
    if (lane == 0) out[w] = word;
    c += (uint32_t)__popc(word);
  }
  if (lane == 0) {
    a.cnt[(size_t)h * a.nb + I] = (int)c;
    const unsigned long long bs = (unsigned long long)a.bs;
    atomicAdd(&a.active[h], (unsigned long long)(c - 1) * bs * bs + bs * (bs + 1) / 2);
  }
}

template <int D, int kBsS>
cudaError_t launch_pass2(const CUtensorMap& mQ, const CUtensorMap& mK, const XaArgs& a, int grid, size_t smem,
                         cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(xattn_score_kernel<D, true, kBsS>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  xattn_score_kernel<D, true, kBsS><<<grid, kXaThreads, smem, s>>>(mQ, mK, a);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_scores(const XaArgs& a, cudaStream_t s) {
  CUtensorMap mQ, mK;
  if (!make_map_strided(&mQ, a.Q, a.R, a.Hq, D, a.S) || !make_map_strided(&mK, a.K, a.R, a.Hkv, D, a.S))
    return cudaErrorInvalidValue;
  const size_t smem = kXaSmem + 1024;
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(xattn_score_kernel<D, false, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)smem)) != cudaSuccess)
    return e;
  const int grid = a.nrt * a.Hq;
  xattn_score_kernel<D, false, 0><<<grid, kXaThreads, smem, s>>>(mQ, mK, a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  switch (a.bsS) {
    case 4: return launch_pass2<D, 4>(mQ, mK, a, grid, smem, s);
    case 8: return launch_pass2<D, 8>(mQ, mK, a, grid, smem, s);
    case 16: return launch_pass2<D, 16>(mQ, mK, a, grid, smem, s);
    case 32: return launch_pass2<D, 32>(mQ, mK, a, grid, smem, s);
    case 64: return launch_pass2<D, 64>(mQ, mK, a, grid, smem, s);
    case 128: return launch_pass2<D, 128>(mQ, mK, a, grid, smem, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_xattn(const XaArgs& a, cudaStream_t s) {
  cudaError_t e;
  // block scores above the diagonal stay zero; the kept-entry counts are sums
  if ((e = cudaMemsetAsync(a.X, 0, (size_t)a.Hq * a.nb * a.nb * sizeof(float), s)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(a.active, 0, (size_t)a.Hq * sizeof(unsigned long long), s)) != cudaSuccess) return e;
  if ((e = (a.d == 128 ? launch_scores<128>(a, s) : launch_scores<64>(a, s))) != cudaSuccess) return e;
  xattn_select_kernel<<<dim3((a.nb + kSelWarps - 1) / kSelWarps, a.Hq), kXaThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace vs
