// Block-sparse causal attention backward: D = rowsum(dO * O) and the
// key-stationary dK / dV kernel (tcgen05).  dQ runs in the query-major
// kernel of attn_fwd.cu.
//
// Gradients of softmax attention with the mask held fixed (ring-attention
// page, section 2.1 online softmax; MTraining review, section
// "分布式稀疏索引近似" active regions):  P = exp(scale S - LSE) on active
// entries, dV = P^T dO, dS = P (dO V^T - D), dK = scale dS^T Q.
//
// Key-stationary tiling.  A work unit keeps 64 keys (K and V rows) in shared
// memory and streams "query sources" = 64 rows (head h, query block I) of
// the GQA group that are active for those keys.  Two sources form a
// 128-row tile (any two: no union waste):
//   S  = Q_tile K^T, dP = dO_tile V^T            M = 128 rows, N = 64 keys
//   P, dS per row (thread per TMEM lane) -> bf16 tiles in shared memory
//   dV^T += dO_tile^T P,  dK^T += Q_tile^T dS    M = d, N = 64 keys, K = rows
// so dK / dV of the 64 keys accumulate in TMEM across all sources and GQA
// heads.  Slash units keep key block kb and stream (h, I) with band
// I/W - kb/W kept (band 0 causal).  Vertical units keep 64 entries of a
// head pair's packed vertical list and stream (h, I) over a slice of the
// later query blocks with per-column masks (vertical m active for rows of
// block I > m/64 whose band is not kept); their fp32 partials are summed,
// in a fixed order, into the slash units' epilogue.
#include "attn_common.cuh"
#include "ptx.cuh"

namespace vs {

namespace {

constexpr int kThreads = 384;
constexpr int kStages = 2;
constexpr int kMaxSplits = 32;

// ---------------------------------------------------------------- D = rowsum(dO * O)
__global__ void bwd_dsum_kernel(const __nv_bfloat16* __restrict__ O, const __nv_bfloat16* __restrict__ dO,
                                float* __restrict__ Dsum, int L, int Hq, int d) {
  // one 16-lane group per (token, head) row; 8 bf16 per lane
  const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long row = gid >> 4;
  const int sub = threadIdx.x & 15;
  float acc = 0.f;
  if (row < (long long)L * Hq) {
    for (int c = sub * 8; c < d; c += 128) {
      const uint4 a = *reinterpret_cast<const uint4*>(O + row * d + c);
      const uint4 b = *reinterpret_cast<const uint4*>(dO + row * d + c);
      const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a);
      const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&b);
      for (int k = 0; k < 4; ++k) {
        const float2 fa = __bfloat1622float2(pa[k]), fb = __bfloat1622float2(pb[k]);
        acc += fa.x * fb.x + fa.y * fb.y;
      }
    }
  }
  for (int o = 8; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (sub == 0 && row < (long long)L * Hq) {
    const int tok = (int)(row / Hq), h = (int)(row % Hq);
    Dsum[(size_t)h * L + tok] = acc;
  }
}

struct BwdParams {
  AttnGeom g;
  const uint32_t* inS;
  const uint32_t* vlist;
  const int32_t* vcnt;
  const int32_t* s_idx;
  const int32_t* s_cnt;
  const float* lse;
  const float* Dsum;
  __nv_bfloat16* dK;
  __nv_bfloat16* dV;
  float* part_k;  // vertical partials [nvg][L][d] (fp32), split slots inside
  float* part_v;
  float* dk32;    // ring steps: fp32 dK / dV sums [L_glob][Hkv][d] that each step adds to
  float* dv32;    // (null: dK / dV written as bf16)
  float scale;
  float log2e;
  DevStatus* status;
  int vertical;   // 1: vertical units, 0: slash units
  int kv_lo, kv_n;  // this launch's key/value heads [kv_lo, kv_lo + kv_n) (one pass)
  int stall;      // bounded-wait test: the planner emits nothing
  // stored dS blocks (null ok: none): see DsPlan
  const int32_t* ds_ok;
  const int32_t* ds_rank;
  const int32_t* ds_base_s;
  const int32_t* ds_base_v;
};

struct SrcMeta {
  int32_t h[2];
  int32_t I[2];
  uint32_t mask[2][2];  // per source, 64 key columns
  int32_t diag[2];      // 1 if the source's rows are the diagonal block of the keys
  int32_t nsrc;
  int32_t first, last;
  int32_t kv0, kv1;     // the unit's stationary keys: packed row (vertical) or (kv head, first key) (slash)
  int32_t blk[2];       // stored dS block of each source (-1: none)
  int32_t pad;
};

// shared memory plan (bytes, 1024-aligned)
constexpr int kHalfRows128 = 128 * 128;  // 128 rows x 128 B
constexpr int kKVs = 0;                  // stationary K (2 x 8 KB) and V (2 x 8 KB): 64 keys
constexpr int kKVsBytes = 4 * 8192;
constexpr int kStage = kKVs + kKVsBytes;
constexpr int kStageBytes = 4 * kHalfRows128;  // Q (2 halves) + dO (2 halves)
constexpr int kPdS = kStage + kStages * kStageBytes;
constexpr int kPdSBytes = 2 * 128 * 128;        // P and dS: 128 rows x 64 keys bf16 each
constexpr int kMQ = 8;  // tile metadata ring (planner -> loader, MMA, P / dS warps)
constexpr int kMeta = kPdS + 2 * kPdSBytes;
constexpr int kBars = kMeta + kMQ * (int)sizeof(SrcMeta);
// kvs_full, kvs_empty, st_full[S], st_empty[S], sdp_full[2], pds_ready[2], pds_free[2], acc_done, acc_free,
// mq_full[MQ], mq_empty[MQ]
constexpr int kNumBars = 2 + 2 * kStages + 6 + 2 + 2 * kMQ;
constexpr int kMisc = kBars + kNumBars * 8;
constexpr int kWaitCyc = kMisc + 64;
constexpr int kSmemBytes = kWaitCyc + kWaitSites * 8;
static_assert(kBars % 8 == 0 && kMisc % 8 == 0 && kWaitCyc % 8 == 0, "mbarriers and counters need 8-byte alignment");

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ bool band_kept(const uint32_t* bm, int B) { return (bm[B >> 5] >> (B & 31)) & 1u; }

// Masking mode of one 64-key block for one source's rows (warp-uniform):
// inactive, fully active, the causal diagonal block, or per-column bits.
enum : int { kSrcOff = 0, kSrcFull = 1, kSrcDiag = 2, kSrcBits = 3 };
__device__ __forceinline__ int src_mode(uint32_t w0, uint32_t w1, bool is_diag) {
  if ((w0 | w1) == 0u) return kSrcOff;
  if (is_diag) return kSrcDiag;
  if ((w0 & w1) == 0xffffffffu) return kSrcFull;
  return kSrcBits;
}
// Active keys of the 64-key block for row rr of its source, as a 64-bit mask.
__device__ __forceinline__ uint64_t active_bits(int mode, uint32_t w0, uint32_t w1, int rr, int strict) {
  if (mode == kSrcOff) return 0ull;
  if (mode == kSrcFull) return ~0ull;
  if (mode == kSrcDiag) return diag_bits(rr, strict);
  return (uint64_t)w0 | ((uint64_t)w1 << 32);
}

// number of row splits of a vertical group and the stride of its partial slots
__device__ __forceinline__ void vsplit(const AttnGeom& g, int cnt, int* R, int* stride) {
  const int r64 = (cnt + 63) & ~63;
  int r = r64 > 0 ? g.L / r64 : 1;
  if (r > kMaxSplits) r = kMaxSplits;
  if (r < 1) r = 1;
  *R = r;
  *stride = r64;
}

// Vertical unit enumeration: units (vg, chunk, split), vg-major, over the
// union groups [vg_lo, vg_hi) of one pass.
struct VUnit {
  int vg, chunk, split, R, stride, cnt;
};
__device__ __forceinline__ int vg_per_kv(const AttnGeom& g) { return g.pair_heads ? g.G / 2 : g.G; }
__device__ bool decode_vunit(const AttnGeom& g, const int32_t* vcnt, int vg_lo, int vg_hi, int id, VUnit* u) {
  for (int vg = vg_lo; vg < vg_hi; ++vg) {
    const int cnt = vcnt[(size_t)vg * (g.nb + 1) + g.nb];
    int R, stride;
    vsplit(g, cnt, &R, &stride);
    const int nchunk = (cnt + 63) / 64;
    const int n = nchunk * R;
    if (id < n) {
      u->vg = vg;
      u->chunk = id / R;
      u->split = id % R;
      u->R = R;
      u->stride = stride;
      u->cnt = cnt;
      return true;
    }
    id -= n;
  }
  return false;
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_dkdv_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mdO,
                     const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mV,
                     const __grid_constant__ CUtensorMap mKp, const __grid_constant__ CUtensorMap mVp,
                     const __grid_constant__ CUtensorMap mDS, const BwdParams P) {
  constexpr int D = 128;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBars);
  uint64_t* kvs_full = bars;
  uint64_t* kvs_empty = bars + 1;
  uint64_t* st_full = bars + 2;
  uint64_t* st_empty = st_full + kStages;
  uint64_t* sdp_full = st_empty + kStages;
  uint64_t* pds_ready = sdp_full + 2;
  // a tile's dV / dK completing frees both its Q / dO stage and its P / dS
  // buffer (both indexed by tile parity), so one commit serves both waiters
  static_assert(kStages == 2, "P / dS buffers and Q / dO stages share the release barrier");
  uint64_t* pds_free = st_empty;
  // stored dS: the loader's store of a tile's dS has read its buffer
  uint64_t* ds_free = pds_ready + 2;
  uint64_t* acc_done = pds_ready + 4;
  uint64_t* acc_free = acc_done + 1;
  uint64_t* mq_full = acc_free + 1;
  uint64_t* mq_empty = mq_full + kMQ;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kMisc + 4);
  // per Q / dO stage, written by the loader before it arms the stage's
  // barrier: nsrc | first << 2 | last << 3 of the stage's tile (the MMA
  // thread's one shared memory load per tile) and the issue clock (profiling)
  volatile uint32_t* stage_word = reinterpret_cast<volatile uint32_t*>(sm + kMisc + 16);
  long long* stage_t = reinterpret_cast<long long*>(sm + kMisc + 32);
  SrcMeta* mq = reinterpret_cast<SrcMeta*>(sm + kMeta);
  unsigned long long* wcyc = reinterpret_cast<unsigned long long*>(sm + kWaitCyc);
  const long long kernel_t0 = clock64();
  const AttnGeom& g = P.g;
  const int W = g.bs / kBlock;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool ds_on = P.ds_ok != nullptr && *P.ds_ok != 0;

  if (threadIdx.x == 0) {
    mbar_init(kvs_full, 1);
    mbar_init(kvs_empty, 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&st_full[i], 1);
      mbar_init(&st_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sdp_full[i], 1);
      mbar_init(&pds_ready[i], 8);  // one arrival per P / dS warp
      mbar_init(&ds_free[i], 1);
    }
    mbar_init(acc_done, 1);
    mbar_init(acc_free, 8);
    for (int i = 0; i < kMQ; ++i) {
      mbar_init(&mq_full[i], 1);
      mbar_init(&mq_empty[i], 9);  // loader, eight P / dS warps
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (threadIdx.x < kWaitSites) wcyc[threadIdx.x] = 0;
  if (warp == 2) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  // TMEM: S[2] at 0, 64; dP[2] at 128, 192; dV^T at 256; dK^T at 320 (64 columns each)
  // a phase that is already complete costs one probe; the abort flag is read
  // only once that probe has failed
  auto wait = [&](uint64_t* bar, uint32_t parity, int where) -> bool {
    const long long w0 = kWaitProfileKv ? clock64() : 0;
    bool ok = mbar_try_wait(bar, parity);
    if (!ok) {
      if (*abort_flag) return false;
      ok = mbar_wait(bar, parity, kWaitLimitNs);
    }
    if (kWaitProfileKv && (threadIdx.x & 31) == 0)
      atomicAdd(&wcyc[where & (kWaitSites - 1)], (unsigned long long)(clock64() - w0));
    if (ok) return true;
    *abort_flag = 1;
    report_timeout_first(P.status, (P.vertical ? kTagDkdvVertical : kTagDkdvSlash) * 100 + where);
    return false;
  };
  // the same, agreed across the warp (callers then issue warp-collective
  // tcgen05 loads/stores, which every lane must execute together)
  auto wait_warp = [&](uint64_t* bar, uint32_t parity, int where) -> bool {
    return __all_sync(0xffffffffu, wait(bar, parity, where));
  };

  // number of units of this launch
  const int vg_lo = P.kv_lo * vg_per_kv(g), vg_hi = (P.kv_lo + P.kv_n) * vg_per_kv(g);
  int nunits;
  if (P.vertical) {
    nunits = 0;
    for (int vg = vg_lo; vg < vg_hi; ++vg) {
      const int cnt = P.vcnt[(size_t)vg * (g.nb + 1) + g.nb];
      int R, stride;
      vsplit(g, cnt, &R, &stride);
      nunits += ((cnt + 63) / 64) * R;
    }
  } else {
    nunits = P.kv_n * g.nb;
  }

  if (warp == 0 && P.stall) {
    // bounded-wait test: the planner emits nothing, so no unit starts and no
    // copy or MMA is ever issued; every other warp's first wait runs out
  } else if (warp == 0) {
    // ------------------------------------------------------------ planner
    // Enumerates each unit's sources, two per tile, into the metadata ring;
    // the loader warp issues the loads, so neither waits on the other's latency.
    const long long prod0 = kWaitProfileKv ? clock64() : 0;
    const uint32_t* bm0 = P.inS;
    const uint32_t* bm1 = P.inS;
    int t = 0;
    for (int uid = blockIdx.x; uid < nunits && !*abort_flag; uid += gridDim.x) {
      int kvh, kb = 0, vg = 0, chunk = 0, split = 0, R = 1, nv = 0;
      int hs[2] = {0, 0};
      int nheads, kv0, kv1 = 0;
      if (P.vertical) {
        VUnit u;
        decode_vunit(g, P.vcnt, vg_lo, vg_hi, uid, &u);
        vg = u.vg;
        chunk = u.chunk;
        split = u.split;
        R = u.R;
        nv = u.cnt;
        if (g.pair_heads) {
          kvh = vg / (g.G / 2);
          hs[0] = kvh * g.G + 2 * (vg % (g.G / 2));
          hs[1] = hs[0] + 1;
          nheads = 2;
        } else {
          kvh = vg / g.G;
          hs[0] = hs[1] = vg;
          nheads = 1;
        }
        bm0 = P.inS + (size_t)hs[0] * g.nw;
        bm1 = P.inS + (size_t)hs[1] * g.nw;
        kv0 = vg * g.L + chunk * 64;
      } else {
        // key blocks in ascending order (more causal rows first)
        kvh = P.kv_lo + uid / g.nb;
        kb = uid % g.nb;
        nheads = g.G;
        kv0 = kvh;
        kv1 = kb * kBlock;
      }

      // ---- the unit's sources, two per tile (warp-uniform registers)
      int nsrc = 0;
      bool first = true;
      int th[2] = {0, 0}, tI[2] = {0, 0}, tdg[2] = {0, 0}, tb[2] = {-1, -1};
      uint32_t tm[2][2] = {{0u, 0u}, {0u, 0u}};
      auto emit = [&](bool last) {
        const int q = t % kMQ;
        bool ok = true;
        if (lane == 0) ok = wait(&mq_empty[q], ((t / kMQ) & 1) ^ 1, 2);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (ok && lane == 0) {
          SrcMeta& m = mq[q];
          m.h[0] = th[0];
          m.h[1] = th[1];
          m.I[0] = tI[0];
          m.I[1] = tI[1];
          m.mask[0][0] = tm[0][0];
          m.mask[0][1] = tm[0][1];
          m.mask[1][0] = tm[1][0];
          m.mask[1][1] = tm[1][1];
          m.diag[0] = tdg[0];
          m.diag[1] = tdg[1];
          m.nsrc = nsrc;
          m.first = first ? 1 : 0;
          m.last = last ? 1 : 0;
          m.kv0 = kv0;
          m.kv1 = kv1;
          m.blk[0] = tb[0];
          m.blk[1] = nsrc > 1 ? tb[1] : -1;
          mbar_arrive(&mq_full[q]);
        }
        __syncwarp();
        ++t;
        nsrc = 0;
        first = false;
      };
      auto put = [&](int h, int I, uint32_t m0, uint32_t m1, int diag, int blk) {
        if (nsrc == 0) {
          th[0] = h;
          tI[0] = I;
          tm[0][0] = m0;
          tm[0][1] = m1;
          tdg[0] = diag;
          tb[0] = blk;
        } else {
          th[1] = h;
          tI[1] = I;
          tm[1][0] = m0;
          tm[1][1] = m1;
          tdg[1] = diag;
          tb[1] = blk;
        }
        ++nsrc;
      };
      // to flag the last tile, a source is placed only once the next one is
      // known (one-source lookahead)
      bool have_look = false;
      int look_h = 0, look_I = 0, look_diag = 0, look_blk = -1;
      uint32_t look_m0 = 0, look_m1 = 0;
      auto push = [&](int h, int I, uint32_t m0, uint32_t m1, int diag, int blk) {
        if (have_look) {
          put(look_h, look_I, look_m0, look_m1, look_diag, look_blk);
          if (nsrc == 2) emit(false);
        }
        have_look = true;
        look_h = h;
        look_I = I;
        look_m0 = m0;
        look_m1 = m1;
        look_diag = diag;
        look_blk = blk;
      };

      if (!P.vertical) {
        for (int hl = 0; hl < nheads && !*abort_flag; ++hl) {
          const int h = kvh * g.G + hl;
          const int ns = P.s_cnt[h];
          bool has0 = false;
          for (int j0 = 0; j0 < ns; j0 += 32) {
            const int j = j0 + lane;
            const int B = (j < ns) ? P.s_idx[(size_t)h * g.nbs + j] : -1;
            if (j0 == 0) has0 = __shfl_sync(0xffffffffu, B, 0) == 0;
            // query blocks of band B for key block kb: I/W = kb/W + B, I >= kb
            const int lo = max(kb, (kb / W + B) * W), hi = min(g.nb - 1, (kb / W + B) * W + W - 1);
            const bool on = B >= 0 && lo <= hi;
            // stored dS: the band's rank and the first block of query block lo
            int rk = 0, b_lo = 0;
            if (ds_on && on) {
              rk = B >= 1 ? P.ds_rank[(size_t)h * g.nbs + B] : 0;
              b_lo = P.ds_base_s[(size_t)h * g.nb + lo];
            }
            uint32_t live = __ballot_sync(0xffffffffu, on);
            while (live) {
              const int k = __ffs(live) - 1;
              live &= live - 1;
              const int lk = __shfl_sync(0xffffffffu, lo, k), hk = __shfl_sync(0xffffffffu, hi, k);
              const int Bk = __shfl_sync(0xffffffffu, B, k), rkk = __shfl_sync(0xffffffffu, rk, k);
              const int bk = __shfl_sync(0xffffffffu, b_lo, k);
              for (int I = lk; I <= hk; ++I) {
                int blk = -1;
                if (ds_on)
                  blk = ds_slash_block(g, I == lk ? bk : P.ds_base_s[(size_t)h * g.nb + I], rkk, Bk, I, kb);
                push(h, I, 0xffffffffu, 0xffffffffu, I == kb ? 1 : 0, blk);
              }
            }
          }
          // band 0 is always active even if the index omits it
          if (!has0) {
            const int lo = kb, hi = min(g.nb - 1, (kb / W) * W + W - 1);
            for (int I = lo; I <= hi; ++I)
              push(h, I, 0xffffffffu, 0xffffffffu, I == kb ? 1 : 0,
                   ds_on ? ds_slash_block(g, P.ds_base_s[(size_t)h * g.nb + I], 0, 0, I, kb) : -1);
          }
        }
      } else {
        // entries [chunk*64, chunk*64 + 64) of the union list; rows of later blocks
        const size_t vbase = (size_t)vg * g.L + chunk * 64;
        const int u0 = chunk * 64 + lane, u1 = u0 + 32;
        const uint32_t e0 = u0 < nv ? P.vlist[vbase + lane] : 0xffffffffu;
        const uint32_t e1 = u1 < nv ? P.vlist[vbase + 32 + lane] : 0xffffffffu;
        const int m0 = u0 < nv ? (int)(e0 & kVTokenMask) : -1;
        const int m1 = u1 < nv ? (int)(e1 & kVTokenMask) : -1;
        const int kbmin = __shfl_sync(0xffffffffu, m0, 0) / kBlock;
        const int Ilo = kbmin + 1;
        const int nI = g.nb - Ilo;
        const int per = (nI + R - 1) / R;
        const int Ib = Ilo + split * per, Ie = min(g.nb, Ib + per);
        for (int hi = 0; hi < nheads; ++hi) {
          const uint32_t* bm = hi ? bm1 : bm0;
          const int h = hs[hi];
          int bv = 0;  // stored dS: first vertical-chunk block of query blocks I0 + lane
          for (int I = Ib; I < Ie && !*abort_flag; ++I) {
            const int I0 = Ib + ((I - Ib) & ~31);
            if (ds_on && I == I0) bv = (I0 + lane < Ie) ? P.ds_base_v[(size_t)h * g.nb + I0 + lane] : 0;
            auto act = [&](int m, uint32_t e) -> bool {
              if (m < 0 || !((e >> (kVFlagShift + hi)) & 1u)) return false;
              const int kbm = m / kBlock;
              if (kbm >= I) return false;
              const int B = I / W - kbm / W;
              return B != 0 && !band_kept(bm, B);
            };
            const uint32_t w0 = __ballot_sync(0xffffffffu, act(m0, e0));
            const uint32_t w1 = __ballot_sync(0xffffffffu, act(m1, e1));
            const int bvI = __shfl_sync(0xffffffffu, bv, I - I0);
            if (w0 | w1) push(h, I, w0, w1, 0, ds_on ? bvI + chunk : -1);
          }
        }
      }
      // flush: the lookahead source is the unit's last
      if (have_look) {
        put(look_h, look_I, look_m0, look_m1, look_diag, look_blk);
        emit(true);
      } else {
        // a vertical unit whose split has no active rows: one empty tile
        put(P.vertical ? hs[0] : kvh * g.G, P.vertical ? g.nb - 1 : kb, 0u, 0u, 0, -1);
        emit(true);
      }
    }
    if (kWaitProfileKv && lane == 0) atomicAdd(&wcyc[28], (unsigned long long)(clock64() - prod0));
  } else if (warp == 3) {
    // ------------------------------------------------------------ loader
    if (lane == 0) {
      int t = 0, un = 0;
      // Stored dS: tile u's dS blocks are stored as soon as the P / dS warps
      // have written them (pds_ready), which the loader meets at tile u + 2
      // before it waits for u's stage; once tile u + 2's loads are issued,
      // the store has read its buffer, and ds_free[u & 1] lets the P / dS
      // warps write it again.  The last two tiles are stored at the end.
      int pblk[2][2] = {{-1, -1}, {-1, -1}};
      // the stored blocks are read back once, after this kernel: evict
      // them first so that the Q / dO tiles keep their place in L2
      const uint64_t pol_stream = ds_on ? l2_policy_evict_first() : 0;
      auto issue_store = [&](int u) -> bool {
        const uint8_t* dbuf = sm + kPdS + (u & 1) * kPdSBytes + 128 * 128;
        bool any = false;
        for (int j = 0; j < 2; ++j)
          if (pblk[u & 1][j] >= 0) {
            tma_store_2d_hint(&mDS, dbuf + j * 8192, 0, pblk[u & 1][j] * 64, pol_stream);
            any = true;
          }
        if (any) bulk_commit_group();
        return any;
      };
      for (int uid = blockIdx.x; uid < nunits && !*abort_flag; uid += gridDim.x, ++un) {
        bool last = false;
        do {
          const int q = t % kMQ;
          if (!wait(&mq_full[q], (t / kMQ) & 1, 3)) break;
          const int nsrc = mq[q].nsrc, kv0 = mq[q].kv0, kv1 = mq[q].kv1;
          const int h0 = mq[q].h[0], h1 = mq[q].h[1], I0 = mq[q].I[0], I1 = mq[q].I[1];
          const int blk0 = mq[q].blk[0], blk1 = mq[q].blk[1];
          const bool first = mq[q].first != 0;
          last = mq[q].last != 0;
          mbar_arrive(&mq_empty[q]);
          if (first) {
            // stationary keys of the unit
            if (!wait(kvs_empty, (un & 1) ^ 1, 1)) break;
            mbar_arrive_expect_tx(kvs_full, kKVsBytes);
            for (int hf = 0; hf < 2; ++hf) {
              if (P.vertical) {
                tma_load_2d(sm + kKVs + hf * 8192, &mKp, kvs_full, hf * 64, kv0);
                tma_load_2d(sm + kKVs + 16384 + hf * 8192, &mVp, kvs_full, hf * 64, kv0);
              } else {
                tma_load_3d(sm + kKVs + hf * 8192, &mK, kvs_full, hf * 64, kv0, kv1);
                tma_load_3d(sm + kKVs + 16384 + hf * 8192, &mV, kvs_full, hf * 64, kv0, kv1);
              }
            }
          }
          bool stored = false;
          if (ds_on && t >= 2) {
            if (!wait(&pds_ready[t & 1], ((t - 2) >> 1) & 1, 6)) break;
            stored = issue_store(t - 2);
          }
          const int st = t % kStages;
          if (!wait(&st_empty[st], ((t / kStages) & 1) ^ 1, 4)) break;
          const long long e0 = kWaitProfileKv ? clock64() : 0;
          uint8_t* qd = sm + kStage + st * kStageBytes;
          uint8_t* od = qd + 2 * kHalfRows128;
          stage_word[st] = (uint32_t)nsrc | (first ? 4u : 0u) | (last ? 8u : 0u);
          if (kWaitProfileKv) stage_t[st] = clock64();
          mbar_arrive_expect_tx(&st_full[st], nsrc * 4 * 8192);
          for (int j = 0; j < nsrc; ++j) {
            const int h = j ? h1 : h0, row = (j ? I1 : I0) * kBlock;
            for (int hf = 0; hf < 2; ++hf) {
              tma_load_3d(qd + hf * kHalfRows128 + j * 8192, &mQ, &st_full[st], hf * 64, h, row);
              tma_load_3d(od + hf * kHalfRows128 + j * 8192, &mdO, &st_full[st], hf * 64, h, row);
            }
          }
          if (kWaitProfileKv) atomicAdd(&wcyc[27], (unsigned long long)(clock64() - e0));
          if (ds_on) {
            if (t >= 2) {
              if (stored) bulk_wait_read_all();
              mbar_arrive(&ds_free[t & 1]);
            }
            pblk[t & 1][0] = blk0;
            pblk[t & 1][1] = blk1;
          }
          ++t;
        } while (!last && !*abort_flag);
      }
      if (ds_on && !*abort_flag) {
        // the last two tiles: wait for their dS, then store
        for (int u = t >= 2 ? t - 2 : 0; u < t; ++u) {
          if (!wait(&pds_ready[u & 1], (u >> 1) & 1, 5)) break;
          issue_store(u);
        }
      }
      if (ds_on) bulk_wait_all();
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescSN64 = idesc_bf16(128, 64, false, false);
      constexpr uint32_t kIdescAcc = idesc_bf16(128, 64, true, true);  // M = d (A^T), N = 64 keys (B MN-major)
      const uint32_t kvs = smem_u32(sm + kKVs);
      // Two kinds of work, issued in whichever order they become ready:
      // S / dP of tile ts (its Q / dO stage landed, fewer than two tiles in
      // flight) and dV / dK of tile ta (its P / dS are in shared memory).
      // Accumulating as soon as P / dS exist frees the tile's stage early, so
      // the next load overlaps the wait for the following tile's data.
      struct Pend {
        int nsrc, first, last, un;
      };
      // Shared memory accesses of this thread wait behind its tcgen05.mma in
      // flight, so the loop keeps its state in registers: the two pending
      // tiles as named variables, the abort flag read only when idle.
      Pend pend0 = {}, pend1 = {};
      int ts = 0, ta = 0;
      int uid = blockIdx.x, un = 0;
      long long idle0 = clock64();
      const long long idle_limit = (long long)(kWaitLimitNs * 21 / 10);
      while (true) {
        const bool more = uid < nunits;
        if (!more && ta == ts) break;
        bool progressed = false;
        const long long i0 = kMmaProfileKv ? clock64() : 0;
        if (ta < ts && mbar_test_wait(&pds_ready[ta & 1], (ta >> 1) & 1)) {
          const Pend q = (ta & 1) ? pend1 : pend0;
          if (q.first && q.un > 0 && !wait(acc_free, (q.un - 1) & 1, 11)) break;
          tc_fence_after();
          const int st = ta % kStages;
          const uint32_t qa = smem_u32(sm + kStage + st * kStageBytes);
          const uint32_t oa = qa + 2 * kHalfRows128;
          const uint32_t pb = smem_u32(sm + kPdS + (ta & 1) * kPdSBytes);
          const uint32_t db = pb + 128 * 128;
          for (int kk = 0; kk < 4 * q.nsrc; ++kk) {
            // rows kk*16 .. kk*16+15: A = dO^T / Q^T (MN-major, two 64-d chunks 16 KB apart)
            const uint32_t acc = (kk > 0 || !q.first) ? 1u : 0u;
            umma_ss(tbase + 256, sdesc_sw128(oa + kk * 2048, kHalfRows128, 1024),
                    sdesc_sw128(pb + kk * 2048, 8192, 1024), kIdescAcc, acc);
            umma_ss(tbase + 320, sdesc_sw128(qa + kk * 2048, kHalfRows128, 1024),
                    sdesc_sw128(db + kk * 2048, 8192, 1024), kIdescAcc, acc);
          }
          umma_commit(&st_empty[st]);  // also the P / dS buffer's release
          if (q.last) umma_commit(acc_done);
          ++ta;
          progressed = true;
          if (kMmaProfileKv) atomicAdd(&wcyc[25], (unsigned long long)(clock64() - i0));
        } else if (more && ts - ta < 2 && mbar_test_wait(&st_full[ts % kStages], (ts / kStages) & 1)) {
          const int st = ts % kStages;
          const uint32_t sw = stage_word[st];
          const struct {
            int nsrc, first, last;
          } m = {(int)(sw & 3u), (int)((sw >> 2) & 1u), (int)((sw >> 3) & 1u)};
          if (kWaitProfileKv) atomicAdd(&wcyc[19], (unsigned long long)(clock64() - stage_t[st]));
          if (m.first && !wait(kvs_full, un & 1, 13)) break;
          tc_fence_after();
          const uint32_t qa = smem_u32(sm + kStage + st * kStageBytes);
          const uint32_t oa = qa + 2 * kHalfRows128;
          const uint32_t buf = (uint32_t)(ts & 1) * 64;
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kHalfRows128 + (kk & 3) * 32;
            const uint32_t koff = (kk >> 2) * 8192 + (kk & 3) * 32;
            umma_ss(tbase + buf, sdesc_sw128(qa + off, 16, 1024), sdesc_sw128(kvs + koff, 16, 1024), kIdescSN64,
                    kk > 0 ? 1u : 0u);
            umma_ss(tbase + 128 + buf, sdesc_sw128(oa + off, 16, 1024), sdesc_sw128(kvs + 16384 + koff, 16, 1024),
                    kIdescSN64, kk > 0 ? 1u : 0u);
          }
          umma_commit(&sdp_full[ts & 1]);
          if (kMmaProfileKv) {
            atomicAdd(&wcyc[16], 1ull);
            atomicAdd(&wcyc[17], (unsigned long long)m.nsrc);
            if (m.last) atomicAdd(&wcyc[18], 1ull);
          }
          // the stationary keys are read only by S and dP: release them now
          if (m.last) umma_commit(kvs_empty);
          if (ts & 1)
            pend1 = Pend{m.nsrc, m.first, m.last, un};
          else
            pend0 = Pend{m.nsrc, m.first, m.last, un};
          ++ts;
          if (m.last) {
            uid += gridDim.x;
            ++un;
          }
          progressed = true;
          if (kMmaProfileKv) atomicAdd(&wcyc[24], (unsigned long long)(clock64() - i0));
        }
        if (progressed) {
          idle0 = clock64();
        } else if (*abort_flag) {
          break;
        } else if (clock64() - idle0 > idle_limit) {
          *abort_flag = 1;
          report_timeout_first(P.status, (P.vertical ? kTagDkdvVertical : kTagDkdvSlash) * 100 + 12);
          break;
        }
      }
    }
    // lanes 1..31 wait here for the issuing lane: the block-wide barrier
    // below is warp-aligned and must see the whole warp together
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ P / dS, epilogue
    // Two warpgroups: group grp owns key columns [32 grp, 32 grp + 32) of every
    // row; thread r of a group owns row r (TMEM lane r).
    const int grp = (threadIdx.x - 128) >> 7;
    const int r = (threadIdx.x - 128) & 127;
    const int src = r >> 6, rr = r & 63;
    const uint32_t lane_off = (uint32_t)(((warp - 4) & 3) * 32) << 16;
    const uint32_t col0 = (uint32_t)(32 * grp);
    int t = 0, un = 0;
    for (int uid = blockIdx.x; uid < nunits && !*abort_flag; uid += gridDim.x, ++un) {
      bool last = false;
      do {
        if (!wait_warp(&mq_full[t % kMQ], (t / kMQ) & 1, 20)) break;
        const SrcMeta& mref = mq[t % kMQ];
        const bool valid = src < mref.nsrc;
        const uint32_t mw0 = valid ? mref.mask[src][0] : 0u, mw1 = valid ? mref.mask[src][1] : 0u;
        const int diag = valid ? mref.diag[src] : 0;
        const int h = mref.h[valid ? src : 0];
        const int tok = mref.I[valid ? src : 0] * kBlock + rr;
        last = mref.last != 0;
        __syncwarp();
        if (lane == 0) mbar_arrive(&mq_empty[t % kMQ]);
        float lse2 = 0.f, Dr = 0.f;
        if (valid && VS_BOUNDS(h < g.Hq && g.tq(tok) < g.L_glob, P.status, 2090)) {
          lse2 = P.lse[(size_t)h * g.L_glob + g.tq(tok)] * P.log2e;
          Dr = P.Dsum[(size_t)h * g.L_glob + g.tq(tok)];
        }
        if (!wait_warp(&sdp_full[t & 1], (t >> 1) & 1, 21)) break;
        const long long ph0 = kWaitProfileKv ? clock64() : 0;
        if (t >= 2 && !wait_warp(&pds_free[t & 1], ((t >> 1) - 1) & 1, 22)) break;
        if (ds_on && t >= 2 && !wait_warp(&ds_free[t & 1], ((t >> 1) - 1) & 1, 9)) break;
        tc_fence_after();
        const float c = P.scale * P.log2e;
        uint8_t* pbuf = sm + kPdS + (t & 1) * kPdSBytes;
        uint8_t* dbuf = pbuf + 128 * 128;
        // warp-uniform masking mode of this row's source for the 64 keys,
        // then this group's 32 of them
        const int mode = src_mode(mw0, mw1, diag != 0);
        const uint32_t act = (uint32_t)(active_bits(mode, mw0, mw1, rr, g.strict_diag) >> col0);
        uint32_t pk[16], dk[16];
        if (mode == kSrcOff) {
#pragma unroll
          for (int k = 0; k < 16; ++k) pk[k] = dk[k] = 0u;
        } else {
          uint32_t sv[32], dv[32];
          const uint32_t tb = tbase + (uint32_t)((t & 1) * 64) + lane_off + col0;
          tmem_ld32(tb, sv);
          tmem_ld32(tb + 128, dv);
          tmem_ld_wait();
          const uint64_t cc = f2pack(c, c), ll = f2pack(-lse2, -lse2);
          if (mode == kSrcFull || act == 0xffffffffu) {
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              float x0, x1, t0, t1;
              ffma2(x0, x1, __uint_as_float(sv[2 * k]), __uint_as_float(sv[2 * k + 1]), cc, ll);
              const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
              pk[k] = pack_bf16(p0, p1);
              fadd2(t0, t1, __uint_as_float(dv[2 * k]), __uint_as_float(dv[2 * k + 1]), -Dr, -Dr);
              fmul2(t0, t1, t0, t1, p0, p1);
              dk[k] = pack_bf16(t0, t1);
            }
          } else {
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              float x0, x1, t0, t1;
              ffma2(x0, x1, __uint_as_float(sv[2 * k]), __uint_as_float(sv[2 * k + 1]), cc, ll);
              const float p0 = ((act >> (2 * k)) & 1u) ? fast_exp2(x0) : 0.f;
              const float p1 = ((act >> (2 * k + 1)) & 1u) ? fast_exp2(x1) : 0.f;
              pk[k] = pack_bf16(p0, p1);
              fadd2(t0, t1, __uint_as_float(dv[2 * k]), __uint_as_float(dv[2 * k + 1]), -Dr, -Dr);
              fmul2(t0, t1, t0, t1, p0, p1);
              dk[k] = pack_bf16(t0, t1);
            }
          }
        }
        // row r of a 128-row x 64-key MN-major SW128 tile: this group's 4 of its 8 chunks of 16 B
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          const int q = 4 * grp + qq;
          const int off = (r >> 3) * 1024 + (r & 7) * 128 + ((q ^ (r & 7)) * 16);
          *reinterpret_cast<uint4*>(pbuf + off) = make_uint4(pk[4 * qq], pk[4 * qq + 1], pk[4 * qq + 2], pk[4 * qq + 3]);
          *reinterpret_cast<uint4*>(dbuf + off) = make_uint4(dk[4 * qq], dk[4 * qq + 1], dk[4 * qq + 2], dk[4 * qq + 3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&pds_ready[t & 1]);
        if (kWaitProfileKv && lane == 0) atomicAdd(&wcyc[26], (unsigned long long)(clock64() - ph0));
        if (last) {
          // ---- epilogue: thread r holds dV^T[d = r][keys of this group] and dK^T likewise
          if (!wait_warp(acc_done, un & 1, 23)) break;
          tc_fence_after();
          const int dcol = r;
          uint32_t av[32], ak[32];
          tmem_ld32(tbase + 256 + lane_off + col0, av);
          tmem_ld32(tbase + 320 + lane_off + col0, ak);
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(acc_free);
          if (P.vertical) {
            VUnit u;
            decode_vunit(g, P.vcnt, vg_lo, vg_hi, uid, &u);
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
              const int e = u.chunk * 64 + (int)col0 + jj;
              if (e < u.cnt && VS_BOUNDS((size_t)u.split * u.stride + e < (size_t)g.L && u.vg < g.nvg, P.status, 2091)) {
                const size_t o = ((size_t)u.vg * g.L + (size_t)u.split * u.stride + e) * D + dcol;
                P.part_v[o] = __uint_as_float(av[jj]);
                P.part_k[o] = __uint_as_float(ak[jj]);
              }
            }
          } else {
            const int kvh = P.kv_lo + uid / g.nb, kb = uid % g.nb;
            // add the vertical partials of tokens in this key block (all union groups of kvh)
            for (int q = 0; q < vg_per_kv(g); ++q) {
              const int vg = kvh * vg_per_kv(g) + q;
              const int cnt = P.vcnt[(size_t)vg * (g.nb + 1) + g.nb];
              int R, stride;
              vsplit(g, cnt, &R, &stride);
              const int e0 = P.vcnt[(size_t)vg * (g.nb + 1) + kb], e1 = P.vcnt[(size_t)vg * (g.nb + 1) + kb + 1];
              for (int e = e0; e < e1; ++e) {
                const int j = (int)(P.vlist[(size_t)vg * g.L + e] & kVTokenMask) - kb * kBlock - (int)col0;
                if (j < 0 || j >= 32) continue;  // the other group's key
                float sk = 0.f, sv = 0.f;
                for (int sp = 0; sp < R; ++sp) {
                  if (!VS_BOUNDS((size_t)sp * stride + e < (size_t)g.L, P.status, 2092)) break;
                  const size_t o = ((size_t)vg * g.L + (size_t)sp * stride + e) * D + dcol;
                  sk += P.part_k[o];
                  sv += P.part_v[o];
                }
#pragma unroll
                for (int jj = 0; jj < 32; ++jj)
                  if (jj == j) {
                    ak[jj] = __float_as_uint(__uint_as_float(ak[jj]) + sk);
                    av[jj] = __float_as_uint(__uint_as_float(av[jj]) + sv);
                  }
              }
            }
            if (P.dk32) {
              // a ring step: add into the fp32 sums of the keys' global rows
#pragma unroll
              for (int jj = 0; jj < 32; ++jj) {
                if (!VS_BOUNDS(g.tk(kb * kBlock + (int)col0 + jj) < g.L_glob && kvh < g.Hkv, P.status, 2093)) break;
                const size_t o = ((size_t)g.tk(kb * kBlock + (int)col0 + jj) * g.Hkv + kvh) * D + dcol;
                P.dv32[o] += __uint_as_float(av[jj]);
                P.dk32[o] += __uint_as_float(ak[jj]) * P.scale;
              }
            } else {
#pragma unroll
              for (int jj = 0; jj < 32; ++jj) {
                if (!VS_BOUNDS(kb * kBlock + (int)col0 + jj < g.L && kvh < g.Hkv, P.status, 2094)) break;
                const size_t o = ((size_t)(kb * kBlock + (int)col0 + jj) * g.Hkv + kvh) * D + dcol;
                P.dV[o] = __float2bfloat16_rn(__uint_as_float(av[jj]));
                P.dK[o] = __float2bfloat16_rn(__uint_as_float(ak[jj]) * P.scale);
              }
            }
          }
        }
        ++t;
      } while (!last && !*abort_flag);
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tbase, 512);
  if (kMmaProfileKv && threadIdx.x < kWaitSites - 1 && wcyc[threadIdx.x])
    atomicAdd(&P.status->wait_cycles[threadIdx.x], wcyc[threadIdx.x]);
  if (kMmaProfileKv && threadIdx.x == kWaitSites - 1) {
    const unsigned long long dt = (unsigned long long)(clock64() - kernel_t0);
    atomicAdd(&P.status->wait_cycles[kWaitSites - 1], dt);
    // the slowest CTA of the slash launch (the tail of the grid)
    if (!P.vertical) atomicMax(&P.status->wait_cycles[kWaitSites - 2], dt);
  }
}

struct BwdWs {
  size_t status, prep_end, dsum, part_k, part_v;
  size_t ds_ok, ds_rank, ds_base_s, ds_base_v, ds;  // stored dS (cap > 0): after everything else
  size_t total;
  PrepWs prep;
};

// cap: stored dS blocks per head (0: none), hpp: query heads per pass
BwdWs bwd_layout(const AttnGeom& g, long long cap, int hpp) {
  WsLayout w;
  BwdWs o;
  o.status = w.take(sizeof(DevStatus));
  o.prep = prep_layout(g, w);
  o.dsum = w.take((size_t)g.Hq * g.L * 4);
  o.part_k = w.take((size_t)g.nvg * g.L * g.d * 4);
  o.part_v = w.take((size_t)g.nvg * g.L * g.d * 4);
  o.ds_ok = o.ds_rank = o.ds_base_s = o.ds_base_v = o.ds = w.off;
  if (cap > 0) {
    o.ds_ok = w.take(4);
    o.ds_rank = w.take((size_t)g.Hq * g.nbs * 4);
    o.ds_base_s = w.take((size_t)g.Hq * g.nb * 4);
    o.ds_base_v = w.take((size_t)g.Hq * g.nb * 4);
    o.ds = w.take(((size_t)hpp * (size_t)cap + 1) * kDsBlockBytes);  // and the zero block
  }
  o.total = w.off;
  return o;
}

// How the stored dS blocks are split: blocks per head and key/value head
// groups per pass (the call runs ceil(Hkv / gpp) passes).
struct DsSplit {
  long long cap = 0;
  int gpp = 1;
};

// Blocks per head that a budget-fill index of density p.density is expected
// to need: density x the causal 64 x 64 blocks of each head, x 1.5 (x 2 for
// the group-shared index, whose unions grow), plus four vertical chunks per
// query block.  0 for top-p selection (no density known in advance).
double ds_blocks_expected(const vs_params& p, const AttnGeom& g) {
  if (!(p.density > 0.f)) return 0.0;
  const double f = p.index_mode == 1 ? 2.0 : 1.5;
  return f * p.density * (double)g.nb * (g.nb + 1) / 2.0 + 4.0 * g.nb;
}

// Block rows of the dS tensor map (hpp cap blocks and the zero block) stay
// below 2^31 (TMA coordinates).
long long ds_row_cap(int hpp) { return (2147483647LL / 64 - 1) / hpp; }

// The split a workspace of ws_bytes allows: one pass over every head when
// the expected blocks fit (or when none are expected: top-p), else the
// fewest passes whose heads each get the expected room, else one key/value
// head group per pass (the most room per head).  The device still checks
// the real counts and recomputes dQ when a head's blocks do not fit.
DsSplit ds_split_for(const vs_params& p, const AttnGeom& g, size_t ws_bytes) {
  DsSplit sp;
  const BwdWs one = bwd_layout(g, 1, 1);
  if (ws_bytes < one.total) return sp;
  const size_t room = ws_bytes - one.ds - kDsBlockBytes;  // less the zero block
  const double want = ds_blocks_expected(p, g);
  for (int n = 1; n <= g.Hkv; ++n) {
    const int gpp = (g.Hkv + n - 1) / n;
    if (n > 1 && gpp == (g.Hkv + n - 2) / (n - 1)) continue;  // the same split as n - 1 passes
    const int hpp = gpp * g.G;
    long long cap = (long long)(room / ((size_t)hpp * kDsBlockBytes));
    if (cap > ds_row_cap(hpp)) cap = ds_row_cap(hpp);
    sp.cap = cap;
    sp.gpp = gpp;
    if (want == 0.0 || (double)cap >= want) break;
  }
  return sp;
}

// Suggested split: every head in one pass up to 32 GiB of blocks; beyond
// that the fewest passes whose blocks take at most 96 GiB; none past that.
DsSplit ds_split_suggested(const vs_params& p, const AttnGeom& g) {
  DsSplit sp;
  const double want = ds_blocks_expected(p, g);
  if (want == 0.0) return sp;
  const long long cap = (long long)want + 1;
  for (int n = 1; n <= g.Hkv; ++n) {
    const int gpp = (g.Hkv + n - 1) / n;
    const int hpp = gpp * g.G;
    const double limit = (n == 1 ? 32.0 : 96.0) * 1024 * 1024 * 1024;
    if ((double)cap * hpp * kDsBlockBytes <= limit && cap <= ds_row_cap(hpp)) {
      sp.cap = cap;
      sp.gpp = gpp;
      return sp;
    }
  }
  return sp;
}

}  // namespace

size_t attn_bwd_ws_bytes(const vs_params& p) { return bwd_layout(make_geom(p), 0, 1).total; }
size_t attn_bwd_ws_bytes_stored(const vs_params& p) {
  const AttnGeom g = make_geom(p);
  const DsSplit sp = ds_split_suggested(p, g);
  return bwd_layout(g, sp.cap, sp.gpp * g.G).total;
}

cudaError_t launch_bwd_dsum(const void* O, const void* dO, float* Dsum, int L, int Hq, int d, cudaStream_t s) {
  const long long rows = (long long)L * Hq;
  const long long threads = rows * 16;
  bwd_dsum_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(
      static_cast<const __nv_bfloat16*>(O), static_cast<const __nv_bfloat16*>(dO), Dsum, L, Hq, d);
  return cudaGetLastError();
}

// dK / dV of the key/value heads [kv_lo, kv_lo + kv_n): the vertical
// launch, then the slash launch
cudaError_t launch_dkdv_heads(const vs_params& p, const AttnGeom& g, const PrepPtrs& pp, const vs_index& ix,
                              const void* Q, const void* K, const void* V, const void* dO, const float* lse,
                              const float* Dsum, void* dK, void* dV, float* part_k, float* part_v, float* dk32,
                              float* dv32, DevStatus* st, const DsPlan* ds, int kv_lo, int kv_n, cudaStream_t s) {
  CUtensorMap mQ, mdO, mK, mV, mKp, mVp, mDS;
  if (kv_lo < 0 || kv_n < 1 || kv_lo + kv_n > g.Hkv) return cudaErrorInvalidValue;
  if (!make_map_heads(&mQ, Q, g.L, g.Hq, 128, g.tq_mul, g.tq_add) ||
      !make_map_heads(&mdO, dO, g.L, g.Hq, 128, g.tq_mul, g.tq_add) ||
      !make_map_heads(&mK, K, g.L, g.Hkv, 128, g.tk_mul, g.tk_add) ||
      !make_map_heads(&mV, V, g.L, g.Hkv, 128, g.tk_mul, g.tk_add) ||
      !make_map_rows(&mKp, pp.Kp, (long long)g.nvg * g.L, 128) ||
      !make_map_rows(&mVp, pp.Vp, (long long)g.nvg * g.L, 128))
    return cudaErrorInvalidValue;
  // the stored dS blocks (a map the kernel never touches when there are none)
  if (ds ? !make_map_rows(&mDS, ds->ds, ((long long)ds->hpp * ds->cap + 1) * 64, 64) : false)
    return cudaErrorInvalidValue;
  if (!ds) mDS = mKp;
  BwdParams P;
  P.g = g;
  P.inS = pp.inS;
  P.vlist = pp.vlist;
  P.vcnt = pp.vcnt;
  P.s_idx = ix.s_idx;
  P.s_cnt = ix.s_cnt;
  P.lse = lse;
  P.Dsum = Dsum;
  P.dK = static_cast<__nv_bfloat16*>(dK);
  P.dV = static_cast<__nv_bfloat16*>(dV);
  P.part_k = part_k;
  P.part_v = part_v;
  P.dk32 = dk32;
  P.dv32 = dv32;
  P.scale = default_scale(p);
  P.log2e = 1.4426950408889634f;
  P.status = st;
  P.kv_lo = kv_lo;
  P.kv_n = kv_n;
  P.stall = test_stall_requested() ? 1 : 0;
  P.ds_ok = ds ? ds->ok : nullptr;
  P.ds_rank = ds ? ds->band_rank : nullptr;
  P.ds_base_s = ds ? ds->base_s : nullptr;
  P.ds_base_v = ds ? ds->base_v : nullptr;
  const size_t smem = kSmemBytes + 1024;
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(attn_dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
      cudaSuccess)
    return e;
  int dev = 0, nsm = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  // vertical units first: their partials feed the slash units' epilogue
  P.vertical = 1;
  attn_dkdv_kernel<<<nsm, kThreads, smem, s>>>(mQ, mdO, mK, mV, mKp, mVp, mDS, P);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  P.vertical = 0;
  const int nunits = kv_n * g.nb;
  attn_dkdv_kernel<<<nunits < nsm ? nunits : nsm, kThreads, smem, s>>>(mQ, mdO, mK, mV, mKp, mVp, mDS, P);
  return cudaGetLastError();
}

cudaError_t launch_dkdv_core(const vs_params& p, const AttnGeom& g, const PrepPtrs& pp, const vs_index& ix,
                             const void* Q, const void* K, const void* V, const void* dO, const float* lse,
                             const float* Dsum, void* dK, void* dV, float* part_k, float* part_v, float* dk32,
                             float* dv32, DevStatus* st, const DsPlan* ds, cudaStream_t s) {
  return launch_dkdv_heads(p, g, pp, ix, Q, K, V, dO, lse, Dsum, dK, dV, part_k, part_v, dk32, dv32, st, ds, 0,
                           g.Hkv, s);
}

size_t bwd_partials_bytes(const AttnGeom& g) { return (size_t)g.nvg * g.L * g.d * 4; }

cudaError_t launch_attn_bwd(const vs_params& p, const vs_index& ix, const void* Q, const void* K, const void* V,
                            const void* O, const float* lse, const void* dO, void* dQ, void* dK, void* dV, void* ws,
                            size_t ws_bytes, cudaStream_t s) {
  if (p.d != 128) return cudaErrorNotSupported;
  const AttnGeom g = make_geom(p);
  const DsSplit sp = ds_split_for(p, g, ws_bytes);
  const long long cap = sp.cap;
  const BwdWs lay = bwd_layout(g, cap, sp.gpp * g.G);
  uint8_t* w = static_cast<uint8_t*>(ws);
  PrepPtrs pp;
  pp.inS = reinterpret_cast<uint32_t*>(w + lay.prep.inS);
  pp.vlist = reinterpret_cast<uint32_t*>(w + lay.prep.vlist);
  pp.vcnt = reinterpret_cast<int32_t*>(w + lay.prep.vcnt);
  pp.Kp = reinterpret_cast<__nv_bfloat16*>(w + lay.prep.Kp);
  pp.Vp = reinterpret_cast<__nv_bfloat16*>(w + lay.prep.Vp);
  pp.vbits = lay.prep.vbits != lay.prep.end ? reinterpret_cast<uint32_t*>(w + lay.prep.vbits) : nullptr;
  float* dsum = reinterpret_cast<float*>(w + lay.dsum);
  DevStatus* st = reinterpret_cast<DevStatus*>(w + lay.status);
  cudaError_t e = launch_attn_prep(g, ix, K, V, pp, s);
  if (e != cudaSuccess) return e;
  if ((e = launch_bwd_dsum(O, dO, dsum, g.L, g.Hq, g.d, s)) != cudaSuccess) return e;
  if (cap == 0) {
    if ((e = launch_dkdv_core(p, g, pp, ix, Q, K, V, dO, lse, dsum, dK, dV,
                              reinterpret_cast<float*>(w + lay.part_k), reinterpret_cast<float*>(w + lay.part_v),
                              nullptr, nullptr, st, nullptr, s)) != cudaSuccess)
      return e;
    if ((e = launch_attn_dq(p, g, pp, Q, K, V, dO, lse, dsum, dQ, st, StepCtl(), s)) != cudaSuccess) return e;
    return p.rope_mode == 1 ? launch_rope_adjoint(p, dQ, dK, nullptr, s) : cudaSuccess;
  }
  // Stored dS: the plan numbers every active block and checks that each
  // head's fit its share of the workspace; per pass (a range of key/value
  // head groups) the dK / dV kernels store them and the dQ kernel reads
  // them back.  If a head's did not fit, the dK / dV kernels store nothing,
  // the reading dQ kernel returns at once, and the recomputing one runs
  // instead (each checks the plan's word).
  DsPlan d;
  d.ok = reinterpret_cast<int32_t*>(w + lay.ds_ok);
  d.band_rank = reinterpret_cast<int32_t*>(w + lay.ds_rank);
  d.base_s = reinterpret_cast<int32_t*>(w + lay.ds_base_s);
  d.base_v = reinterpret_cast<int32_t*>(w + lay.ds_base_v);
  d.ds = reinterpret_cast<__nv_bfloat16*>(w + lay.ds);
  d.cap = (int)cap;
  d.hpp = sp.gpp * g.G;
  d.zero_blk = d.hpp * d.cap;
  if ((e = cudaMemsetAsync(d.ds + (size_t)d.zero_blk * 64 * 64, 0, kDsBlockBytes, s)) != cudaSuccess) return e;
  if ((e = launch_ds_plan(g, pp, d, s)) != cudaSuccess) return e;
  for (int kv_lo = 0; kv_lo < g.Hkv; kv_lo += sp.gpp) {
    const int kv_n = g.Hkv - kv_lo < sp.gpp ? g.Hkv - kv_lo : sp.gpp;
    if ((e = launch_dkdv_heads(p, g, pp, ix, Q, K, V, dO, lse, dsum, dK, dV,
                               reinterpret_cast<float*>(w + lay.part_k), reinterpret_cast<float*>(w + lay.part_v),
                               nullptr, nullptr, st, &d, kv_lo, kv_n, s)) != cudaSuccess)
      return e;
    if ((e = launch_dq_stored(p, g, pp, K, d, dQ, st, kv_lo, kv_n, s)) != cudaSuccess) return e;
  }
  StepCtl ctl;
  ctl.skip_if = d.ok;
  if ((e = launch_attn_dq(p, g, pp, Q, K, V, dO, lse, dsum, dQ, st, ctl, s)) != cudaSuccess) return e;
  // rope_mode = 1: the stored-dS dQ kernel applied the RoPE adjoint in its
  // epilogue; the recomputing one did not, so dQ's pass runs only when the
  // plan chose that path (its word is then zero)
  return p.rope_mode == 1 ? launch_rope_adjoint(p, dQ, dK, d.ok, s) : cudaSuccess;
}

}  // namespace vs
