// Sparse-index approximation, selection stage, and the exact active-entry
// count.  One CTA per query head.
//
// MTraining review, section "分布式稀疏索引近似": keep the minimum number of
// vertical lines and slash bands that recall the target attention mass
// ("online top-p budget" in the training-loss section).  Reading: each
// direction independently keeps the smallest prefix of its masses sorted in
// descending order (ties: lower index first) whose sum reaches top_p of the
// direction's total; band 0 is always kept.  top_p >= 1 keeps every element
// with positive mass.
//
// Budget-fill variant (the experiments fix sparsity at 95 %, section 八
// item 4): verticals and bands >= 1 are ranked together by mass (both
// directions total last_q) and the kept set is band 0 plus every candidate
// with mass >= tau, tau the largest value whose set reaches the requested
// active density.
//
// Selection by threshold: masses are non-negative fp32, so their bit
// patterns order like the values.  A most-significant-digit-first radix
// descent (11/11/10 bits) over a histogram of counts and masses finds the
// threshold key; masses are summed as exact 64-bit fixed-point integers
// (scale 2^sh, sum < 2^62), so every sum is order-independent and the
// selection is deterministic.  Kept elements are then compacted in index
// order, which yields ascending lists.
//
// Active entries (section 四 "核心公式" sparsity ratio): band B >= 1 covers
// (nbs - B) full bs x bs tiles, band 0 the causal halves of the nbs diagonal
// tiles, and a kept vertical m adds bs entries for each later row tile whose
// band is not kept.
#include <cuda_bf16.h>

#include "common.cuh"

namespace vs {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;

struct SelShared {
  unsigned long long hsum[2048];
  unsigned int hcnt[2048];
  unsigned long long wsum[kWarps];
  unsigned int wcnt[kWarps];
  unsigned int wcnt2[kWarps];
  unsigned long long bcast_u64[4];
  unsigned int bcast_u32[4];
};

__device__ __forceinline__ uint32_t key_of(float x) { return __float_as_uint(x); }

__device__ __forceinline__ unsigned long long quant(float x, int sh) {
  // exact x * 2^sh (power-of-two scale), truncated to an integer
  return (unsigned long long)__float2ull_rz(ldexpf(x, sh));
}

// Block-wide sum (all threads get the result).
__device__ unsigned long long block_sum_u64(unsigned long long v, SelShared& sh) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) sh.wsum[warp] = v;
  __syncthreads();
  unsigned long long t = 0;
  for (int w = 0; w < kWarps; ++w) t += sh.wsum[w];
  __syncthreads();
  return t;
}

// Largest key tau such that sum of quantised masses of elements with key >= tau
// reaches `target` (target >= 1).  Also returns the mass/count strictly above
// tau and the count/mass at tau.
struct Thresh {
  uint32_t tau;
  unsigned long long sum_gt;
  unsigned int cnt_gt;
  unsigned int cnt_eq;
  unsigned long long qtau;
};

__device__ Thresh radix_threshold(const float* x, int n, int sh, unsigned long long target, SelShared& s) {
  uint32_t prefix = 0, pmask = 0;
  unsigned long long above = 0;
  unsigned int above_cnt = 0, eq_cnt = 0;
  const int shifts[3] = {21, 10, 0};
  const int bits[3] = {11, 11, 10};
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = shifts[pass], nb = 1 << bits[pass];
    for (int b = threadIdx.x; b < nb; b += kThreads) {
      s.hsum[b] = 0;
      s.hcnt[b] = 0;
    }
    __syncthreads();
    for (int base = 0; base < n; base += kThreads) {
      const int i = base + threadIdx.x;
      float xv = 0.f;
      bool in = false;
      uint32_t k = 0;
      if (i < n) {
        xv = x[i];
        k = key_of(xv);
        in = (k & pmask) == prefix;
      }
      const int bin = in ? (int)((k >> shift) & (uint32_t)(nb - 1)) : -1;
      // aggregate equal bins within the warp before touching shared memory;
      // the 61-bit masses are summed in three 21-bit parts (no overflow)
      const unsigned same = __match_any_sync(0xffffffffu, bin);
      if (in) {
        const unsigned long long q = quant(xv, sh);
        const unsigned s0 = __reduce_add_sync(same, (unsigned)(q & 0x1FFFFFull));
        const unsigned s1 = __reduce_add_sync(same, (unsigned)((q >> 21) & 0x1FFFFFull));
        const unsigned s2 = __reduce_add_sync(same, (unsigned)(q >> 42));
        if ((__ffs(same) - 1) == (int)(threadIdx.x & 31)) {
          atomicAdd(&s.hsum[bin], (unsigned long long)s0 + ((unsigned long long)s1 << 21) +
                                      ((unsigned long long)s2 << 42));
          atomicAdd(&s.hcnt[bin], (unsigned)__popc(same));
        }
      }
    }
    __syncthreads();
    // suffix sums from the top bin down, done by warp 0
    if (threadIdx.x < 32) {
      const int lane = threadIdx.x;
      const int per = nb / 32;  // contiguous bins per lane (64 or 32)
      unsigned long long ls = 0;
      unsigned lc = 0;
      for (int b = lane * per; b < (lane + 1) * per; ++b) {
        ls += s.hsum[b];
        lc += s.hcnt[b];
      }
      // exclusive suffix over lanes: mass of all bins above this lane's range
      unsigned long long suf = ls;
      unsigned sufc = lc;
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long t = __shfl_down_sync(0xffffffffu, suf, o);
        const unsigned tc = __shfl_down_sync(0xffffffffu, sufc, o);
        if (lane + o < 32) {
          suf += t;
          sufc += tc;
        }
      }
      const unsigned long long above_lane = suf - ls;  // bins strictly above my range
      const unsigned above_lane_c = sufc - lc;
      // the lane whose range contains the crossing
      const bool hit = (above + above_lane < target) && (above + suf >= target);
      const unsigned hb = __ballot_sync(0xffffffffu, hit);
      int chosen_lane = hb ? (__ffs(hb) - 1) : -1;
      if (chosen_lane < 0) chosen_lane = 0;  // target beyond total: take everything
      if (lane == chosen_lane) {
        unsigned long long acc = above + above_lane;
        unsigned accc = above_lane_c;
        int bsel = lane * per;
        for (int b = (lane + 1) * per - 1; b >= lane * per; --b) {
          if (acc + s.hsum[b] >= target || b == lane * per) {
            bsel = b;
            break;
          }
          acc += s.hsum[b];
          accc += s.hcnt[b];
        }
        s.bcast_u64[0] = acc;
        s.bcast_u32[0] = above_cnt + accc;
        s.bcast_u32[1] = (uint32_t)bsel;
        s.bcast_u32[2] = s.hcnt[bsel];
      }
    }
    __syncthreads();
    above = s.bcast_u64[0];
    above_cnt = s.bcast_u32[0];
    prefix |= s.bcast_u32[1] << shift;
    pmask |= (uint32_t)(nb - 1) << shift;
    eq_cnt = s.bcast_u32[2];
    __syncthreads();
  }
  Thresh t;
  t.tau = prefix;
  t.sum_gt = above;
  t.cnt_gt = above_cnt;
  t.cnt_eq = eq_cnt;
  t.qtau = quant(__uint_as_float(prefix), sh);
  return t;
}

// Compact {i : key_i > tau} plus the first `n_tie` indices with key_i == tau,
// in index order, into out[]; returns the count.  If accum_vert is set, also
// returns (via *vert_entries) the sum over kept i of bs * notS[nbs-1-i/bs].
__device__ int compact_select(const float* x, int n, uint32_t tau, unsigned n_tie, int32_t* out,
                              const int32_t* notS, int nbs, int bs, unsigned long long* vert_entries,
                              SelShared& s, int skip_index) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int base = 0;
  unsigned tie_base = 0;
  unsigned long long ve = 0;
  for (int start = 0; start < n; start += kThreads) {
    const int i = start + threadIdx.x;
    bool gt = false, eq = false;
    if (i < n && i != skip_index) {
      const uint32_t k = key_of(x[i]);
      gt = k > tau;
      eq = k == tau;
    }
    const unsigned bgt = __ballot_sync(0xffffffffu, gt);
    const unsigned beq = __ballot_sync(0xffffffffu, eq);
    if (lane == 0) {
      s.wcnt[warp] = __popc(bgt);
      s.wcnt2[warp] = __popc(beq);
    }
    __syncthreads();
    unsigned tie_before = 0, eq_total = 0;
    for (int w = 0; w < kWarps; ++w) {
      if (w < warp) tie_before += s.wcnt2[w];
      eq_total += s.wcnt2[w];
    }
    const unsigned lanemask = (1u << lane) - 1u;
    const unsigned my_tie_rank = tie_base + tie_before + __popc(beq & lanemask);
    const bool keep = gt || (eq && my_tie_rank < n_tie);
    const unsigned bkeep = __ballot_sync(0xffffffffu, keep);
    __syncthreads();
    if (lane == 0) s.wcnt[warp] = __popc(bkeep);
    __syncthreads();
    int before = 0, total = 0;
    for (int w = 0; w < kWarps; ++w) {
      if (w < warp) before += s.wcnt[w];
      total += s.wcnt[w];
    }
    if (keep) {
      out[base + before + __popc(bkeep & lanemask)] = i;
      if (notS) ve += (unsigned long long)bs * (unsigned long long)notS[nbs - 1 - i / bs];
    }
    base += total;
    tie_base += eq_total;
    __syncthreads();
  }
  if (vert_entries) *vert_entries = block_sum_u64(ve, s);
  return base;
}

// The same compaction for {i : key_i > tau} alone (no ties) over a 16-byte
// aligned x with n a multiple of 4: each thread takes four consecutive
// elements per pass, a warp scan and one scan of the warp totals place them.
__device__ int compact_above(const float* x, int n, uint32_t tau, int32_t* out, const int32_t* notS, int nbs,
                             int bs, unsigned long long* vert_entries, SelShared& s) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float4* x4 = reinterpret_cast<const float4*>(x);
  int base = 0;
  unsigned long long ve = 0;
  for (int start = 0; start < n / 4; start += kThreads) {
    const int q = start + threadIdx.x;
    bool k0 = false, k1 = false, k2 = false, k3 = false;
    if (q < n / 4) {
      const float4 v = x4[q];
      k0 = key_of(v.x) > tau;
      k1 = key_of(v.y) > tau;
      k2 = key_of(v.z) > tau;
      k3 = key_of(v.w) > tau;
    }
    const int cnt = (int)k0 + (int)k1 + (int)k2 + (int)k3;
    int incl = cnt;
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) s.wcnt[warp] = (unsigned)incl;
    __syncthreads();
    if (warp == 0) {
      const int w = (int)s.wcnt[lane];
      int wi = w;
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, wi, o);
        if (lane >= o) wi += t;
      }
      s.wcnt2[lane] = (unsigned)(wi - w);
      if (lane == 31) s.bcast_u32[3] = (unsigned)wi;
    }
    __syncthreads();
    int o = base + (int)s.wcnt2[warp] + incl - cnt;
    const int total = (int)s.bcast_u32[3];
    if (cnt) {
      const int i0 = 4 * q;
      if (notS) ve += (unsigned long long)bs * (unsigned long long)cnt * (unsigned long long)notS[nbs - 1 - i0 / bs];
      if (k0) out[o++] = i0;
      if (k1) out[o++] = i0 + 1;
      if (k2) out[o++] = i0 + 2;
      if (k3) out[o++] = i0 + 3;
    }
    base += total;
  }
  if (vert_entries) *vert_entries = block_sum_u64(ve, s);
  return base;
}

// notS[x] = #{B in [1, x] : B not kept}; kept given by inS (0/1 per band).
// Block-wide scan: each thread counts a run of consecutive bands, the warps
// scan their threads' counts, warp 0 the warps' totals.
__device__ void build_notS(const uint8_t* inS, int32_t* notS, int nbs, SelShared& s) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int per = (nbs + kThreads - 1) / kThreads;
  const int b0 = threadIdx.x * per;
  int cnt = 0;
  for (int j = 0; j < per; ++j) {
    const int b = b0 + j;
    if (b >= 1 && b < nbs && !inS[b]) ++cnt;
  }
  int incl = cnt;
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) s.wcnt[warp] = (unsigned)incl;
  __syncthreads();
  if (warp == 0) {
    const int w = (int)s.wcnt[lane];
    int wi = w;
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += t;
    }
    s.wcnt2[lane] = (unsigned)(wi - w);  // bands counted by the warps before this one
  }
  __syncthreads();
  int run = (int)s.wcnt2[warp] + incl - cnt;  // not-kept bands before this thread's run
  for (int j = 0; j < per; ++j) {
    const int b = b0 + j;
    if (b < nbs) {
      if (b >= 1 && !inS[b]) ++run;
      notS[b] = run;
    }
  }
  __syncthreads();
}

__device__ unsigned long long slash_entries(const uint8_t* inS, int nbs, int bs, SelShared& s) {
  unsigned long long e = 0;
  for (int B = threadIdx.x; B < nbs; B += kThreads) {
    if (!inS[B]) continue;
    e += (B == 0) ? (unsigned long long)nbs * (unsigned long long)(bs * (bs + 1) / 2)
                  : (unsigned long long)(nbs - B) * (unsigned long long)bs * (unsigned long long)bs;
  }
  return block_sum_u64(e, s);
}

// Budget fill: verticals whose key reached the running threshold, gathered in
// shared memory once they fit, so later threshold probes skip the full list.
constexpr int kCandCap = 8192;
// budget fill, fast path: verticals gathered above a histogram cut
constexpr int kFastCap = 1024;
// and the search warps' kept-band tables (bits and word prefixes)
constexpr int kWarpTables = 32 * 1024;

__global__ void __launch_bounds__(kThreads, 1) select_kernel(const IndexArgs a) {
  extern __shared__ __align__(16) uint8_t dyn[];
  __shared__ SelShared s;
  const int h = blockIdx.x;
  const int nbs = a.nbs, L = a.L, bs = a.bs;
  uint8_t* inS = dyn;                                               // [nbs]
  int32_t* notS = reinterpret_cast<int32_t*>(dyn + align_up(nbs, 16));  // [nbs]
  uint32_t* ckey = reinterpret_cast<uint32_t*>(dyn + align_up(nbs, 16) + align_up((size_t)nbs * 4, 16));
  int32_t* cblk = reinterpret_cast<int32_t*>(ckey + kCandCap);  // candidate list: key, key block
  const float* v = a.v + (size_t)h * L;
  const float* S = a.S + (size_t)h * nbs;
  int32_t* vout = a.v_idx + (size_t)h * L;
  int32_t* sout = a.s_idx + (size_t)h * nbs;
  // fixed-point scale: masses are <= last_q, so last_q * 2^sh < 2^62
  int lg = 0;
  while ((1 << lg) < a.last_q + 1) ++lg;
  const int sh = 61 - lg;

  unsigned long long slash_e = 0, vert_e = 0;
  int nv = 0, ns = 0;
  if (a.density <= 0.f) {
    // ---------------- top-p, slash direction
    unsigned long long tot = 0;
    for (int B = threadIdx.x; B < nbs; B += kThreads) tot += quant(S[B], sh);
    tot = block_sum_u64(tot, s);
    uint32_t tau;
    unsigned ntie;
    if (a.top_p >= 1.f || tot == 0) {
      tau = 1;  // every positive mass (key >= smallest positive denormal)
      ntie = 0xffffffffu;
      // keys > tau are kept; key == tau (the smallest denormal) kept too
    } else {
      unsigned long long target = (unsigned long long)((double)a.top_p * (double)tot);
      if ((double)target < (double)a.top_p * (double)tot) ++target;
      if (target < 1) target = 1;
      const Thresh t = radix_threshold(S, nbs, sh, target, s);
      tau = t.tau;
      unsigned long long need = target > t.sum_gt ? target - t.sum_gt : 0;
      unsigned long long k = t.qtau ? (need + t.qtau - 1) / t.qtau : 1;
      if (k < 1) k = 1;
      if (k > t.cnt_eq) k = t.cnt_eq;
      ntie = (unsigned)k;
    }
    for (int B = threadIdx.x; B < nbs; B += kThreads) inS[B] = 0;
    __syncthreads();
    // compaction writes ascending band ids; band 0 forced separately
    ns = compact_select(S, nbs, tau, ntie, sout, nullptr, nbs, bs, nullptr, s, -1);
    // mark kept bands, then force band 0 in (keeping the list ascending)
    for (int j = threadIdx.x; j < ns; j += kThreads) inS[sout[j]] = 1;
    __syncthreads();
    if (!inS[0]) {
      // shift right by one and put 0 first (single thread; ns <= nbs - 1 here)
      if (threadIdx.x == 0) {
        for (int j = ns; j > 0; --j) sout[j] = sout[j - 1];
        sout[0] = 0;
      }
      __syncthreads();
      if (threadIdx.x == 0) inS[0] = 1;
      ++ns;
    }
    __syncthreads();
    build_notS(inS, notS, nbs, s);
    slash_e = slash_entries(inS, nbs, bs, s);
    // ---------------- top-p, vertical direction
    tot = 0;
    for (int m = threadIdx.x; m < L; m += kThreads) tot += quant(v[m], sh);
    tot = block_sum_u64(tot, s);
    if (a.top_p >= 1.f || tot == 0) {
      tau = 1;
      ntie = 0xffffffffu;
    } else {
      unsigned long long target = (unsigned long long)((double)a.top_p * (double)tot);
      if ((double)target < (double)a.top_p * (double)tot) ++target;
      if (target < 1) target = 1;
      const Thresh t = radix_threshold(v, L, sh, target, s);
      tau = t.tau;
      unsigned long long need = target > t.sum_gt ? target - t.sum_gt : 0;
      unsigned long long k = t.qtau ? (need + t.qtau - 1) / t.qtau : 1;
      if (k < 1) k = 1;
      if (k > t.cnt_eq) k = t.cnt_eq;
      ntie = (unsigned)k;
    }
    nv = compact_select(v, L, tau, ntie, vout, notS, nbs, bs, &vert_e, s, -1);
  } else {
    // ---------------- budget fill
    const double T = (double)L * (double)(L + 1) * 0.5;
    const unsigned long long target = (unsigned long long)ceil((double)a.density * T);
    // Verticals with key >= the accepted threshold, once there are at most
    // kCandCap of them: the threshold only rises, so later probes need no
    // other vertical (ncand < 0: not gathered yet, probe the full list).
    int ncand = -1;
    unsigned long long nabove = 0;  // verticals with key >= the last probed threshold
    auto entries_at = [&](uint32_t tau) -> unsigned long long {
      for (int B = threadIdx.x; B < nbs; B += kThreads) inS[B] = (B == 0) || (key_of(S[B]) >= tau);
      __syncthreads();
      build_notS(inS, notS, nbs, s);
      const unsigned long long se = slash_entries(inS, nbs, bs, s);
      unsigned long long ve = 0, c = 0;
      if (ncand < 0) {
        // four verticals per 16-byte load (L and bs are multiples of 64, so
        // the four share a key block)
        const float4* v4 = reinterpret_cast<const float4*>(v);
#pragma unroll 4
        for (int q = threadIdx.x; q < L / 4; q += kThreads) {
          const float4 x = v4[q];
          const unsigned n4 = (key_of(x.x) >= tau) + (key_of(x.y) >= tau) + (key_of(x.z) >= tau) +
                              (key_of(x.w) >= tau);
          if (n4) {
            ve += (unsigned long long)n4 * (unsigned long long)notS[nbs - 1 - (4 * q) / bs];
            c += n4;
          }
        }
      } else {
        for (int i = threadIdx.x; i < ncand; i += kThreads)
          if (ckey[i] >= tau) {
            ve += (unsigned long long)notS[nbs - 1 - cblk[i]];
            ++c;
          }
      }
      // the block totals stay below 2^34 (ve) and 2^21 (c): one block sum carries both
      const unsigned long long both = block_sum_u64((ve << 21) | c, s);
      nabove = both & ((1ull << 21) - 1ull);
      return se + (both >> 21) * (unsigned long long)bs;
    };
    auto gather = [&](uint32_t tau) {
      if (ncand >= 0 || nabove > (unsigned long long)kCandCap) return;
      if (threadIdx.x == 0) s.bcast_u32[0] = 0u;
      __syncthreads();
      for (int m0 = 0; m0 < L; m0 += kThreads) {
        // one shared-memory atomic per warp (L is a multiple of 64)
        const int m = m0 + (int)threadIdx.x;
        const uint32_t k = m < L ? key_of(v[m]) : 0u;
        const bool in = m < L && k >= tau;
        const unsigned b = __ballot_sync(0xffffffffu, in);
        unsigned i0 = 0;
        if ((threadIdx.x & 31) == 0 && b) i0 = atomicAdd(&s.bcast_u32[0], (unsigned)__popc(b));
        i0 = __shfl_sync(0xffffffffu, i0, 0);
        if (in) {
          const unsigned i = i0 + (unsigned)__popc(b & ((1u << (threadIdx.x & 31)) - 1u));
          ckey[i] = k;
          cblk[i] = m / bs;
        }
      }
      __syncthreads();
      ncand = (int)s.bcast_u32[0];
      __syncthreads();
    };
    // Fast path.  A cut t_low from a histogram of the vertical keys (2048
    // bins of key >> 20): the lowest bin edge with at most kFastCap
    // verticals at or above it.  Those verticals are gathered in index
    // order; if the set at t_low reaches the target, tau >= t_low and only
    // they matter: seven warps finish the search three bits per round
    // (warp_entries) and the kept verticals are compacted from them.
    // Otherwise the bitwise search over the full list runs.
    long long pf[8] = {};
    const long long pf0 = kProfileSel ? clock64() : 0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (a.vhist) {
      // counted by the scoring pass
      for (int b = threadIdx.x; b < 2048; b += kThreads) s.hcnt[b] = a.vhist[(size_t)h * 2048 + b];
    } else {
      for (int b = threadIdx.x; b < 2048; b += kThreads) s.hcnt[b] = 0u;
      __syncthreads();
      // four keys per thread and step, the steps' loads issued together
      const float4* v4 = reinterpret_cast<const float4*>(v);
      const int L4 = L / 4;
      for (int q0 = 0; q0 < L4; q0 += 4 * kThreads) {
        float4 x[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int q = q0 + u * kThreads + (int)threadIdx.x;
          x[u] = q < L4 ? v4[q] : make_float4(-1.f, -1.f, -1.f, -1.f);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float xs[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            // negative: past the end (keys of masses are below 2^31)
            const int bin = xs[j] < 0.f ? -1 : (int)min(key_of(xs[j]) >> 20, 2047u);
            const unsigned same = __match_any_sync(0xffffffffu, bin);
            if (bin >= 0 && (__ffs(same) - 1) == lane) atomicAdd(&s.hcnt[bin], (unsigned)__popc(same));
          }
        }
      }
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // suffix counts over the bins, 64 per lane from the top
      unsigned c = 0;
      for (int b = lane * 64; b < lane * 64 + 64; ++b) c += s.hcnt[b];
      unsigned suf = c;
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned t = __shfl_down_sync(0xffffffffu, suf, o);
        if (lane + o < 32) suf += t;
      }
      // lanes whose whole range fits: the one below the lowest of them
      // refines bin by bin
      const unsigned fits = __ballot_sync(0xffffffffu, suf <= (unsigned)kFastCap);
      const int l0 = fits ? __ffs(fits) - 1 : 32;
      int cut = l0 * 64;
      if (l0 > 0 && lane == l0 - 1) {
        unsigned acc = suf - c;  // bins above this lane's range
        int b = lane * 64 + 64;
        while (b > lane * 64 && acc + s.hcnt[b - 1] <= (unsigned)kFastCap) {
          acc += s.hcnt[b - 1];
          --b;
        }
        cut = b;
      }
      cut = __shfl_sync(0xffffffffu, cut, l0 > 0 ? l0 - 1 : 0);
      if (lane == 0) s.bcast_u32[1] = (unsigned)cut << 20;
    }
    __syncthreads();
    const uint32_t t_low = s.bcast_u32[1];
    if (kProfileSel) pf[0] = clock64() - pf0;
    // The verticals with key >= t_low (at most kFastCap by the cut) and the
    // bands >= 1 with key >= t_low, gathered in any order.  Slots of the
    // candidate arrays: [0, kFastCap) the verticals (key, token), then their
    // working copy (key, band row x = nbs - 1 - key block), then the bands'
    // working list (key, band).  After each search round the working lists
    // keep only keys above tau: later thresholds are all above it.
    uint32_t* ckey2 = ckey;
    int32_t* cidx = cblk;
    uint32_t* wkey = ckey + kFastCap;
    int32_t* wx = cblk + kFastCap;
    uint32_t* bkey = ckey + 2 * kFastCap;
    int32_t* bidx = cblk + 2 * kFastCap;
    constexpr int kBandCap = kCandCap - 2 * kFastCap;
    int nw = 0, nbc = 0;
    bool fast = false;
    // warp-aggregated slot in a shared counter
    auto slot = [&](bool in, unsigned* counter) -> unsigned {
      const unsigned bal = __ballot_sync(0xffffffffu, in);
      unsigned i0 = 0;
      if (lane == 0 && bal) i0 = atomicAdd(counter, (unsigned)__popc(bal));
      return __shfl_sync(0xffffffffu, i0, 0) + (unsigned)__popc(bal & ((1u << lane) - 1u));
    };
    if (t_low < 0x7f800000u) {
      if (threadIdx.x == 0) {
        s.bcast_u32[2] = 0u;
        s.bcast_u32[3] = 0u;
      }
      __syncthreads();
      // four 16-byte loads (16 verticals) per thread in flight per step (v is
      // 16-byte aligned and L a multiple of 64)
      const float4* v4 = reinterpret_cast<const float4*>(v);
      const int L4 = L / 4;
      for (int q0 = 0; q0 < L4; q0 += 4 * kThreads) {
        float4 x[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int q = q0 + u * kThreads + (int)threadIdx.x;
          x[u] = q < L4 ? v4[q] : make_float4(-1.f, -1.f, -1.f, -1.f);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int m4 = 4 * (q0 + u * kThreads + (int)threadIdx.x);
          const float xs[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            // negative: past the end (keys of masses are below 2^31)
            const bool in = xs[j] >= 0.f && key_of(xs[j]) >= t_low;
            const unsigned i = slot(in, &s.bcast_u32[2]);
            if (in && i < (unsigned)kFastCap) {
              ckey2[i] = key_of(xs[j]);
              cidx[i] = m4 + j;
              wkey[i] = key_of(xs[j]);
              wx[i] = nbs - 1 - (m4 + j) / bs;
            }
          }
        }
      }
      for (int B0 = 0; B0 < nbs; B0 += kThreads) {
        const int B = B0 + (int)threadIdx.x;
        const uint32_t k = B < nbs ? key_of(S[B]) : 0u;
        const bool in = B >= 1 && B < nbs && k >= t_low;
        const unsigned i = slot(in, &s.bcast_u32[3]);
        if (in && i < (unsigned)kBandCap) {
          bkey[i] = k;
          bidx[i] = B;
        }
      }
      __syncthreads();
      ncand = (int)s.bcast_u32[2];
      nbc = (int)s.bcast_u32[3];
      nw = ncand;
      __syncthreads();
      if (ncand > kFastCap || nbc > kBandCap) ncand = -1;  // cannot hold them: the full search
    }
    if (kProfileSel) {
      pf[2] = clock64() - pf0 - pf[0];
      pf[6] = ncand;
    }
    const int nwords = (nbs + 31) / 32;
    // search warps: as many as the tables fit, up to 31 (2^nbr - 1 thresholds per round)
    int nsw = kWarpTables / (8 * nwords);
    if (nsw > 32) nsw = 32;
    int nbr = 0;
    while ((2 << nbr) - 1 <= nsw - 1 && nbr < 5) ++nbr;  // 2^nbr - 1 evaluators (warps 1..)
    uint32_t* wbm = reinterpret_cast<uint32_t*>(cblk + kCandCap);  // [nsw][nwords] kept-band bits
    int32_t* wpre = reinterpret_cast<int32_t*>(wbm + nsw * nwords);  // [nsw][nwords] kept bands in earlier words
    const unsigned long long band0 = (unsigned long long)nbs * (unsigned long long)(bs * (bs + 1) / 2);
    // active entries at threshold t, by one warp over the working lists
    auto warp_entries = [&](uint32_t t) -> unsigned long long {
      uint32_t* bm = wbm + warp * nwords;
      int32_t* pre = wpre + warp * nwords;
      unsigned long long se = 0;
      // kept bands: the working ones with key >= t
      for (int wd = lane; wd < nwords; wd += 32) bm[wd] = 0u;
      __syncwarp();
      for (int i = lane; i < nbc; i += 32)
        if (bkey[i] >= t) {
          const int B = bidx[i];
          atomicOr(&bm[B >> 5], 1u << (B & 31));
          se += (unsigned long long)(nbs - B) * (unsigned long long)bs * (unsigned long long)bs;
        }
      __syncwarp();
      int carry = 0;
      for (int base = 0; base < nwords; base += 32) {
        const int wd = base + lane;
        const int c = wd < nwords ? __popc(bm[wd]) : 0;
        int incl = c;
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        if (wd < nwords) pre[wd] = carry + incl - c;
        carry += __shfl_sync(0xffffffffu, incl, 31);
      }
      __syncwarp();
      unsigned long long ve = 0;
      // not-kept bands in [1, x] for each vertical at or above t
      for (int i = lane; i < nw; i += 32) {
        const int x = wx[i];
        if (wkey[i] < t || x < 1) continue;
        const int w = x >> 5, j = x & 31;
        const uint32_t msk = j == 31 ? 0xffffffffu : ((2u << j) - 1u);
        ve += (unsigned long long)(x - (pre[w] + __popc(bm[w] & msk)));
      }
      for (int o = 16; o > 0; o >>= 1) {
        se += __shfl_xor_sync(0xffffffffu, se, o);
        ve += __shfl_xor_sync(0xffffffffu, ve, o);
      }
      return band0 + se + ve * (unsigned long long)bs;
    };
    uint32_t tau = 0u;
    if (ncand >= 0 && nbr >= 1) {
      fast = true;
      bool first_round = true;
      for (int hi = 30; hi >= 0; hi -= nbr) {
        const int nbit = hi >= nbr - 1 ? nbr : hi + 1;
        const int lo = hi - nbit + 1;
        if (warp < (1 << nbit)) {
          if (warp == 0) {
            // the set at t_low must reach the target (checked beside the first search round)
            if (first_round) {
              const bool ok = warp_entries(t_low) >= target;
              if (lane == 0) s.bcast_u64[3] = ok ? 1ull : 0ull;  // a slot nothing else writes
            }
          } else {
            const uint32_t cand = tau | ((uint32_t)warp << lo);
            // monotone: every threshold at or below t_low reaches the target
            const bool ok = cand <= 0x7f800000u && (cand <= t_low || warp_entries(cand) >= target);
            if (lane == 0) s.wcnt[warp] = ok ? 1u : 0u;
          }
        }
        __syncthreads();
        if (first_round && s.bcast_u64[3] == 0ull) {
          fast = false;  // (read by every thread before the next barrier; the slot is not reused)
          break;
        }
        first_round = false;
        unsigned k = 0;
        for (int w = 1; w < (1 << nbit); ++w)
          if (s.wcnt[w]) k = (unsigned)w;
        tau |= k << lo;
        // working lists: keys above tau only (one vertical, up to six bands per thread)
        uint32_t vk = 0u, bk[6];
        int vx = 0, bb[6];
        const int i = (int)threadIdx.x;
        if (i < nw) {
          vk = wkey[i];
          vx = wx[i];
        }
#pragma unroll
        for (int u = 0; u < 6; ++u) {
          const int j = u * kThreads + i;
          bk[u] = j < nbc ? bkey[j] : 0u;
          bb[u] = j < nbc ? bidx[j] : 0;
        }
        if (threadIdx.x == 0) {
          s.bcast_u32[2] = 0u;
          s.bcast_u32[3] = 0u;
        }
        __syncthreads();
        {
          const bool in = i < nw && vk > tau;
          const unsigned p = slot(in, &s.bcast_u32[2]);
          if (in) {
            wkey[p] = vk;
            wx[p] = vx;
          }
        }
#pragma unroll
        for (int u = 0; u < 6; ++u) {
          const bool in = u * kThreads + i < nbc && bk[u] > tau;
          const unsigned p = slot(in, &s.bcast_u32[3]);
          if (in) {
            bkey[p] = bk[u];
            bidx[p] = bb[u];
          }
        }
        __syncthreads();
        nw = (int)s.bcast_u32[2];
        nbc = (int)s.bcast_u32[3];
        __syncthreads();
      }
      if (tau == 0u) tau = 1u;  // every positive candidate
      if (kProfileSel) {
        pf[3] = clock64() - pf0 - pf[0] - pf[2];
        pf[5] = fast ? 1 : 0;
      }
    }
    if (!fast) {
      // the bitwise search, probing the whole vertical list until its
      // candidates fit the gathered list
      ncand = -1;
      if (entries_at(0x7f800001u) >= target) {
        tau = 0x7f800001u;  // nothing beyond band 0
      } else if (entries_at(1u) < target) {
        tau = 1u;  // every positive candidate
      } else {
        tau = 0u;
        for (int bit = 30; bit >= 0; --bit) {
          const uint32_t cand = tau | (1u << bit);
          if (cand > 0x7f800000u) continue;
          if (entries_at(cand) >= target) {
            tau = cand;
            gather(tau);
          }
        }
      }
    }
    // final sets at tau: slash list (band 0 forced) and verticals
    for (int B = threadIdx.x; B < nbs; B += kThreads) inS[B] = (B == 0) || (key_of(S[B]) >= tau);
    __syncthreads();
    build_notS(inS, notS, nbs, s);
    slash_e = slash_entries(inS, nbs, bs, s);
    // bands: keep key >= tau, i.e. key > tau - 1 ... use compaction with tie = all
    ns = compact_select(S, nbs, tau - 1u, 0u, sout, nullptr, nbs, bs, nullptr, s, 0);
    // band 0 forced: it was skipped above (skip_index = 0); prepend it
    if (threadIdx.x == 0) {
      for (int j = ns; j > 0; --j) sout[j] = sout[j - 1];
      sout[0] = 0;
    }
    __syncthreads();
    ++ns;
    if (fast) {
      // the kept verticals are gathered candidates (any order): each is
      // placed by the number of kept tokens below it
      int32_t* kept = wx;  // free after the search
      if (threadIdx.x == 0) s.bcast_u32[2] = 0u;
      __syncthreads();
      for (int c0 = 0; c0 < ncand; c0 += kThreads) {
        const int i = c0 + (int)threadIdx.x;
        const bool in = i < ncand && ckey2[i] >= tau;
        const unsigned p = slot(in, &s.bcast_u32[2]);
        if (in) kept[p] = cidx[i];
      }
      __syncthreads();
      const int K = (int)s.bcast_u32[2];
      unsigned long long ve = 0;
      for (int i = threadIdx.x; i < K; i += kThreads) {
        const int e = kept[i];
        int pos = 0;
        for (int j = 0; j < K; ++j) pos += kept[j] < e ? 1 : 0;
        vout[pos] = e;
        ve += (unsigned long long)bs * (unsigned long long)notS[nbs - 1 - e / bs];
      }
      vert_e = block_sum_u64(ve, s);
      nv = K;
    } else {
      nv = compact_above(v, L, tau - 1u, vout, notS, nbs, bs, &vert_e, s);
    }
    if (kProfileSel && threadIdx.x == 0 && a.status) {
      pf[4] = clock64() - pf0;
      for (int k = 0; k < 7; ++k) atomicAdd(&a.status->wait_cycles[k], (unsigned long long)pf[k]);
    }
  }
  if (threadIdx.x == 0) {
    a.v_cnt[h] = nv;
    a.s_cnt[h] = ns;
    if (a.active) a.active[h] = (long long)(slash_e + vert_e);
  }
}

}  // namespace

// kept-band flags, band prefix table, budget-fill candidate list (key, block)
// (and, after them, each search warp's kept-band bits and word prefixes)
size_t select_smem_bytes(int nbs) {
  return align_up(nbs, 16) + align_up((size_t)nbs * 4, 16) + (size_t)kCandCap * 8 + kWarpTables + (size_t)kFastCap * 2;
}

cudaError_t launch_select(const IndexArgs& a, cudaStream_t s) {
  const size_t smem = select_smem_bytes(a.nbs);
  cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  select_kernel<<<a.Hq, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace vs
