// dQ of the sparse attention backward from stored dS tiles.
//
// MTraining review, section 三/核心创新/2 (compute only the non-zero regions of
// each sub-matrix) and the ring-attention page, section 2.1 (the gradient of
// one query row is a sum over its KV blocks): dQ_i = scale * sum over the
// active keys m of row i of dS_im k_m.  The key-stationary dK / dV kernel
// already forms every active 64 x 64 block of dS = P (dP - D); when the
// workspace has room it also stores them (bf16), and this kernel streams them
// back with the matching key tiles: one tcgen05 product dQ += dS K per pair of
// key sources, no recomputation of S and dP.  The blocks cost 2 bytes per
// active entry written and read once; the work left is 2 d FLOP per entry.
//
// The row tiles, their key sources and the per-segment masks are those of the
// query-major kernel (two 64-row segments, slash key blocks in descending
// order, then 64-entry chunks of the vertical union list); a source that is
// inactive for a segment gets zeros in that segment's rows of the dS tile.
#include "attn_common.cuh"
#include "ptx.cuh"

namespace vs {
namespace {

// ------------------------------------------------------------------ plan

// block-wide exclusive scan of one int per thread (blockDim.x a multiple of
// 32, at most 1024); returns the block total
__device__ int plan_block_scan(int x, int* excl, int* wsum) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarp = blockDim.x >> 5;
  int incl = x;
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  int before = 0, total = 0;
  for (int k = 0; k < nwarp; ++k) {
    if (k < warp) before += wsum[k];
    total += wsum[k];
  }
  __syncthreads();
  *excl = before + incl - x;
  return total;
}

// One CTA per query head: the rank of every kept band, then the number of
// dS blocks of each query block (its slash sources and vertical chunks) and
// their exclusive scan.  A head whose blocks exceed the capacity clears *ok.
__global__ void __launch_bounds__(1024) ds_plan_kernel(AttnGeom g, const uint32_t* __restrict__ inS,
                                                      const int32_t* __restrict__ vcnt, DsPlan d) {
  __shared__ int wsum[32];
  __shared__ int carry;
  const int h = blockIdx.x;
  const int vg = g.pair_heads ? h / 2 : h;
  const int W = g.bs / kBlock;
  const uint32_t* bm = inS + (size_t)h * g.nw;
  int32_t* rank = d.band_rank + (size_t)h * g.nbs;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < g.nbs; base += blockDim.x) {
    const int B = base + threadIdx.x;
    const int k = (B >= 1 && B < g.nbs && ((bm[B >> 5] >> (B & 31)) & 1u)) ? 1 : 0;
    int excl;
    const int tot = plan_block_scan(k, &excl, wsum);
    const int c0 = carry;
    if (B < g.nbs) rank[B] = c0 + excl + k;
    __syncthreads();
    if (threadIdx.x == 0) carry = c0 + tot;
    __syncthreads();
  }
  // the ranks written above are read back by other threads of this block
  __threadfence_block();
  __syncthreads();
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  const long long head0 = (long long)(h % d.hpp) * d.cap;
  for (int base = 0; base < g.nb; base += blockDim.x) {
    const int I = base + threadIdx.x;
    int n = 0, ns = 0;
    if (I < g.nb) {
      const int Iw = I / W;
      ns = (I - Iw * W + 1) + W * rank[Iw];
      n = ns + (vcnt[(size_t)vg * (g.nb + 1) + I] + 63) / 64;
    }
    int excl;
    const int tot = plan_block_scan(n, &excl, wsum);
    const int c0 = carry;
    if (I < g.nb) {
      d.base_s[(size_t)h * g.nb + I] = (int32_t)(head0 + c0 + excl);
      d.base_v[(size_t)h * g.nb + I] = (int32_t)(head0 + c0 + excl + ns);
    }
    __syncthreads();
    if (threadIdx.x == 0) carry = c0 + tot;
    __syncthreads();
  }
  if (threadIdx.x == 0 && carry > d.cap) atomicExch(d.ok, 0);
}

// ------------------------------------------------------------------ dQ

struct DqsParams {
  AttnGeom g;
  const uint32_t* inS;
  const uint32_t* vlist;
  const int32_t* vcnt;
  const int32_t* base_s;
  const int32_t* base_v;
  const int32_t* ok;
  __nv_bfloat16* dq;
  int zero_blk;     // the block of zeros
  int kv_lo, kv_n;  // this pass: the row tiles of key/value heads [kv_lo, kv_lo + kv_n)
  int nitems;       // their number
  float scale;
  DevStatus* status;
  // RoPE adjoint fused into the epilogue (rope_mode = 1): channel i pairs
  // with i + 64 and is rotated by -t theta_i, t the row's token
  int32_t rope;
  float rope_mscale;
  uint64_t rope_turn[64];  // theta_i / (2 pi) as 0.64 fixed-point fractions
};

constexpr int kQsThreads = 256;  // warp 0 planner, 1 MMA, 2 tensor memory, 3 loader, 4..7 epilogue
constexpr int kQsStages = 3;
constexpr int kHalf = 128 * 128;        // 128 rows x 128 bytes
constexpr int kStageA = 0;              // dS: per source [128 rows x 64 keys] (segment 0 rows, then segment 1)
constexpr int kStageB = 2 * kHalf;      // K: per d half [128 keys x 64 d] (source 0 keys, then source 1)
constexpr int kStageBytes = 4 * kHalf;  // 64 KB
constexpr int kWordOff = kQsStages * kStageBytes;  // per stage: nsrc | first << 2 | last << 3
constexpr int kRecs = 8;                            // planner -> loader record ring
constexpr int kRecOff = kWordOff + 64;
constexpr int kBarOff = kRecOff + kRecs * 32;
// full[S], empty[S], acc_done[2], acc_free[2], rec_full[R], rec_empty[R]
constexpr int kNumBars = 2 * kQsStages + 4 + 2 * kRecs;
constexpr int kMiscOff = kBarOff + kNumBars * 8;  // tensor memory slot, abort flag
constexpr int kQsSmem = kMiscOff + 16;

__device__ __forceinline__ bool kept(const uint32_t* bm, int B) { return (bm[B >> 5] >> (B & 31)) & 1u; }

// One tile of two key sources (the second absent when nsrc = 1).
struct TileRec {
  int32_t src0, src1;  // slash: key block; vertical: -1 - packed row of the chunk
  int32_t b00, b01;    // dS block of source 0 for segment 0 / 1 (-1: zeros)
  int32_t b10, b11;    // the same for source 1
  int32_t kvh;         // key/value head of the slash K tiles
  uint32_t word;       // nsrc | first << 2 | last << 3; 0 ends the stream
};
static_assert(sizeof(TileRec) == 32, "record slots are 32 bytes");

__global__ void __launch_bounds__(kQsThreads, 1)
    dq_stored_kernel(const __grid_constant__ CUtensorMap mDS, const __grid_constant__ CUtensorMap mK,
                     const __grid_constant__ CUtensorMap mKp, const DqsParams P) {
  // the stored tiles did not fit: the recomputing dQ kernel runs instead
  if (*P.ok == 0) return;
  // one thread of one launch at a time (the passes run in stream order)
  if (blockIdx.x == 0 && threadIdx.x == 0 && P.status) {
    P.status->path = 1;
    P.status->passes += 1;
  }
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBarOff);
  uint64_t* full = bars;
  uint64_t* empty = full + kQsStages;
  uint64_t* acc_done = empty + kQsStages;
  uint64_t* acc_free = acc_done + 2;
  uint64_t* rec_full = acc_free + 2;
  uint64_t* rec_empty = rec_full + kRecs;
  volatile uint32_t* word = reinterpret_cast<volatile uint32_t*>(sm + kWordOff);
  volatile TileRec* recs = reinterpret_cast<volatile TileRec*>(sm + kRecOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kMiscOff + 4);
  const AttnGeom& g = P.g;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // profiling build (VS_WAIT_PROFILE=7): cycles per part, added into the
  // status block's wait_cycles by lane 0 of each role's warp at the end
  long long pc[8] = {};
  const long long k0 = kWaitProfileDs ? clock64() : 0;
  auto tick = [&]() -> long long { return kWaitProfileDs ? clock64() : 0; };

  if (threadIdx.x == 0) {
    for (int i = 0; i < kQsStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_done[i], 1);
      mbar_init(&acc_free[i], 4);  // one arrival per epilogue warp
    }
    for (int i = 0; i < kRecs; ++i) {
      mbar_init(&rec_full[i], 1);
      mbar_init(&rec_empty[i], 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, 256);  // two 128-column dQ accumulators
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
    report_timeout_first(P.status, kTagDqStored * 100 + where);
    return false;
  };
  auto wait_warp = [&](uint64_t* bar, uint32_t parity, int where) -> bool {
    return __all_sync(0xffffffffu, wait(bar, parity, where));
  };

  if (warp == 0) {
    // ------------------------------------------------------------ planner
    // Walks each row tile's key sources and writes one record per pair of
    // sources into the record ring; a record with word 0 ends the stream.
    const int W = g.bs / kBlock;
    const long long pl0 = tick();
    int t = 0;
    auto put_rec = [&](uint32_t wd, int s0, int s1, int b00, int b01, int b10, int b11, int kvh) -> bool {
      const int q = t % kRecs;
      bool ok = true;
      if (lane == 0) {
        const long long r0 = tick();
        ok = wait(&rec_empty[q], ((t / kRecs) & 1) ^ 1, 1);
        if (kWaitProfileDs) pc[1] += tick() - r0;
        if (ok) {
          volatile TileRec& r = recs[q];
          r.src0 = s0;
          r.src1 = s1;
          r.b00 = b00;
          r.b01 = b01;
          r.b10 = b10;
          r.b11 = b11;
          r.kvh = kvh;
          r.word = wd;
          mbar_arrive(&rec_full[q]);
        }
      }
      ++t;
      return __shfl_sync(0xffffffffu, ok, 0);
    };
    for (int id = blockIdx.x; id < P.nitems && !*abort_flag; id += gridDim.x) {
      const long long h0 = tick();
      // the item in scalars (an indexed struct would live in local memory)
      const Item it = decode_item_kv(g, id, P.kv_lo, P.kv_n);
      const int I0 = it.I[0], I1 = it.I[1], kvh = it.g, vg = it.vg;
      const bool val0 = it.valid[0], val1 = it.valid[1];
      const uint32_t* bm0 = P.inS + (size_t)it.h[0] * g.nw;
      const uint32_t* bm1 = P.inS + (size_t)it.h[1] * g.nw;
      const int Itop = val1 ? max(I0, I1) : I0;
      const int Iw = I0 / W;
      // the row's first slash / vertical blocks and its vertical count,
      // loaded together
      const size_t r0 = (size_t)it.h[0] * g.nb + I0;
      const size_t r1 = (size_t)it.h[1] * g.nb + (val1 ? I1 : I0);
      const int bsl0 = P.base_s[r0], bvt0 = P.base_v[r0];
      const int bsl1 = P.base_s[r1], bvt1 = P.base_v[r1];
      const int nv = P.vcnt[(size_t)vg * (g.nb + 1) + Itop];
      int run0 = 0, run1 = 0;  // slash blocks of each segment so far
      auto slash_active = [&](int s, int kb) -> bool {
        const int Is = s ? I1 : I0;
        if (!(s ? val1 : val0) || kb < 0 || kb > Is) return false;
        const int B = Is / W - kb / W;
        return B == 0 || kept(s ? bm1 : bm0, B);
      };
      // kept-band words of the two segments for bands 32 w .. 32 w + 31 up
      // to the diagonal band Iw (band 0 forced); head-paired tiles only
      auto band_words = [&](int w, uint32_t* u0, uint32_t* u1) {
        *u0 = *u1 = 0u;
        if (w * 32 > Iw) return;
        uint32_t x = bm0[w], y = bm1[w];
        const int top = Iw - w * 32;
        if (top < 31) {
          x &= (2u << top) - 1u;
          y &= (2u << top) - 1u;
        }
        if (w == 0) {
          x |= 1u;
          y |= 1u;
        }
        *u0 = x;
        *u1 = y;
      };
      // ---- count the sources first so the row tile's last one is flagged
      int nslash = 0;
      if (g.pair_heads) {
        int cnt = 0;
        for (int w0 = 0; w0 * 32 <= Iw; w0 += 32) {
          uint32_t u0, u1;
          band_words(w0 + lane, &u0, &u1);
          cnt += __popc((u0 | u1) & (w0 + lane == 0 ? ~1u : ~0u));
        }
        nslash = __reduce_add_sync(0xffffffffu, cnt) * W + (I0 - Iw * W + 1);
      } else {
        for (int kb0 = Itop; kb0 >= 0; kb0 -= 32) {
          const int kb = kb0 - lane;
          nslash += __popc(__ballot_sync(0xffffffffu, slash_active(0, kb) || slash_active(1, kb)));
        }
      }
      const int nchunks = (nv + 63) / 64;
      const int total_src = nslash + nchunks;
      if (kWaitProfileDs) pc[2] += tick() - h0;

      // the pending source (at most one; a second completes a tile)
      int nsrc = 0, done = 0;
      bool first = true, ok = true;
      int ps = 0, pb0 = -1, pb1 = -1;
      auto push = [&](int src, int b0, int b1) {
        if (nsrc == 0) {
          ps = src;
          pb0 = b0;
          pb1 = b1;
          nsrc = 1;
          if (done + 1 < total_src) return;
          done += 1;
          ok = put_rec(1u | (first ? 4u : 0u) | 8u, ps, 0, pb0, pb1, -1, -1, kvh) && ok;
        } else {
          done += 2;
          const bool last = done == total_src;
          ok = put_rec(2u | (first ? 4u : 0u) | (last ? 8u : 0u), ps, src, pb0, pb1, b0, b1, kvh) && ok;
        }
        nsrc = 0;
        first = false;
      };
      // ---- slash sources: bands ascending, key blocks descending
      if (g.pair_heads) {
        for (int w0 = 0; w0 * 32 <= Iw && ok; w0 += 32) {
          uint32_t u0, u1;
          band_words(w0 + lane, &u0, &u1);
          uint32_t nz = __ballot_sync(0xffffffffu, (u0 | u1) != 0u);
          while (nz) {
            const int jw = __ffs(nz) - 1;
            nz &= nz - 1;
            const uint32_t a0 = __shfl_sync(0xffffffffu, u0, jw), a1 = __shfl_sync(0xffffffffu, u1, jw);
            uint32_t u = a0 | a1;
            while (u) {
              const int bit = __ffs(u) - 1;
              u &= u - 1;
              const int B = (w0 + jw) * 32 + bit;
              const int lo = (Iw - B) * W, hi = min(I0, lo + W - 1);
              const bool on0 = (a0 >> bit) & 1u, on1 = (a1 >> bit) & 1u;
              for (int kbs = hi; kbs >= lo; --kbs) push(kbs, on0 ? bsl0 + run0++ : -1, on1 ? bsl1 + run1++ : -1);
            }
          }
        }
      } else {
        for (int kb0 = Itop; kb0 >= 0 && ok; kb0 -= 32) {
          const int kb = kb0 - lane;
          const uint32_t c0 = __ballot_sync(0xffffffffu, slash_active(0, kb));
          const uint32_t c1 = __ballot_sync(0xffffffffu, slash_active(1, kb));
          uint32_t u = c0 | c1;
          while (u) {
            const int bit = __ffs(u) - 1;
            u &= u - 1;
            const bool on0 = (c0 >> bit) & 1u, on1 = (c1 >> bit) & 1u;
            push(kb0 - bit, on0 ? bsl0 + run0++ : -1, on1 ? bsl1 + run1++ : -1);
          }
        }
      }
      // ---- vertical sources: 64-entry chunks of the union list below block Itop
      for (int c = 0; c < nchunks && ok; ++c) {
        bool act0 = false, act1 = false;
        for (int half = 0; half < 2; ++half) {
          const int u = c * 64 + half * 32 + lane;
          if (u < nv) {
            const uint32_t e = P.vlist[(size_t)vg * g.L + u];
            const int kbm = (int)(e & kVTokenMask) / kBlock;
            const uint32_t f = e >> kVFlagShift;
            if (val0 && (f & 1u) && kbm < I0) {
              const int B = I0 / W - kbm / W;
              act0 = act0 || (B != 0 && !kept(bm0, B));
            }
            if (val1 && ((f >> 1) & 1u) && kbm < I1) {
              const int B = I1 / W - kbm / W;
              act1 = act1 || (B != 0 && !kept(bm1, B));
            }
          }
        }
        const bool any0 = __any_sync(0xffffffffu, act0), any1 = __any_sync(0xffffffffu, act1);
        push(-1 - (vg * g.L + c * 64), any0 ? bvt0 + c : -1, any1 ? bvt1 + c : -1);
      }
      if (!ok) break;
    }
    if (!*abort_flag) put_rec(0u, 0, 0, -1, -1, -1, -1, 0);  // end of the stream
    if (kWaitProfileDs && lane == 0) {
      pc[0] = tick() - pl0;
      for (int k = 0; k < 3; ++k) atomicAdd(&P.status->wait_cycles[k], (unsigned long long)pc[k]);
    }
  } else if (warp == 3) {
    // ------------------------------------------------------------ loader
    // One tile per record: the TMA loads of its dS blocks (the block of
    // zeros for a segment the source does not reach) and of its K tiles.
    if (lane == 0) {
      tma_prefetch_desc(&mDS);
      tma_prefetch_desc(&mK);
      tma_prefetch_desc(&mKp);
    }
    const long long ld0 = tick();
    const uint64_t pol_stream = l2_policy_evict_first(), pol_keep = l2_policy_evict_last();
    for (int t = 0;; ++t) {
      const int q = t % kRecs;
      bool ok = true;
      const long long r0 = tick();
      if (lane == 0) ok = wait(&rec_full[q], (t / kRecs) & 1, 2);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      __syncwarp();  // lane 0's acquire orders the other lanes' reads too
      const volatile TileRec& r = recs[q];
      const uint32_t wd = r.word;
      const int s0 = r.src0, s1 = r.src1, kvh = r.kvh;
      const int b00 = r.b00, b01 = r.b01, b10 = r.b10, b11 = r.b11;
      __syncwarp();
      if (lane == 0) mbar_arrive(&rec_empty[q]);
      if (wd == 0u) break;
      const int nsrc = (int)(wd & 3u);
      const int st = t % kQsStages;
      if (lane == 0) ok = wait(&empty[st], ((t / kQsStages) & 1) ^ 1, 4);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      __syncwarp();
      const long long e1 = tick();
      if (kWaitProfileDs) pc[3] += e1 - r0;
      uint8_t* a = sm + st * kStageBytes + kStageA;
      uint8_t* bb = sm + st * kStageBytes + kStageB;
      if (kWaitProfileDs) pc[5] += (int)(b00 < 0) + (int)(b01 < 0) + (nsrc > 1 ? (int)(b10 < 0) + (int)(b11 < 0) : 0);
      if (lane == 0) {
        word[st] = wd;
        mbar_arrive_expect_tx(&full[st], (uint32_t)(4 * nsrc) * 8192u);
      }
      __syncwarp();
      // one copy per lane: lanes 0-3 the dS blocks (source l / 2, segment
      // l % 2), lanes 4-7 the K tiles (source (l - 4) / 2, d half l % 2)
      // the dS blocks are read once (evict first); K tiles, re-read by
      // every row tile whose sources include them, and the block of zeros
      // stay (evict last)
      if (lane < 8) {
        const int j = (lane >> 1) & 1, k = lane & 1;
        if (j < nsrc) {
          if (lane < 4) {
            const int blk = j ? (k ? b11 : b10) : (k ? b01 : b00);
            tma_load_2d_hint(a + j * kHalf + k * 8192, &mDS, &full[st], 0, (blk >= 0 ? blk : P.zero_blk) * 64,
                             blk >= 0 ? pol_stream : pol_keep);
          } else {
            const int src = j ? s1 : s0;
            uint8_t* kd = bb + k * kHalf + j * 8192;
            if (src >= 0)
              tma_load_3d_hint(kd, &mK, &full[st], k * 64, kvh, src * kBlock, pol_keep);
            else
              tma_load_2d_hint(kd, &mKp, &full[st], k * 64, -1 - src, pol_keep);
          }
        }
      }
      __syncwarp();
      if (kWaitProfileDs) {
        pc[4] += tick() - e1;
        pc[6] += 1;
      }
    }
    if (kWaitProfileDs && lane == 0) {
      pc[7] = tick() - ld0;
      for (int k = 3; k < 8; ++k) atomicAdd(&P.status->wait_cycles[k], (unsigned long long)pc[k]);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdesc = idesc_bf16(128, 128, false, true);  // A = dS K-major, B = K MN-major
      int t = 0, it_local = 0;
      for (int id = blockIdx.x; id < P.nitems && !*abort_flag; id += gridDim.x, ++it_local) {
        const int b = it_local & 1;
        const uint32_t tacc = tbase + (uint32_t)(b * 128);
        const long long f0 = tick();
        if (it_local >= 2 && !wait(&acc_free[b], ((it_local >> 1) - 1) & 1, 11)) break;
        if (kWaitProfileDs) pc[1] += tick() - f0;
        bool last = false;
        do {
          const int st = t % kQsStages;
          const long long w0 = tick();
          if (!wait(&full[st], (t / kQsStages) & 1, 12)) break;
          const long long w1 = tick();
          if (kWaitProfileDs) pc[0] += w1 - w0;
          const uint32_t w = word[st];
          const int nsrc = (int)(w & 3u);
          const bool first = (w >> 2) & 1u;
          last = (w >> 3) & 1u;
          tc_fence_after();
          const uint64_t ad0 = sdesc_sw128(smem_u32(sm + st * kStageBytes + kStageA), 16, 1024);
          const uint64_t bd0 = sdesc_sw128(smem_u32(sm + st * kStageBytes + kStageB), kHalf, 1024);
          for (int kk = 0; kk < 4 * nsrc; ++kk)
            umma_ss(tacc, sdesc_add(ad0, (kk >> 2) * kHalf + (kk & 3) * 32), sdesc_add(bd0, kk * 2048), kIdesc,
                    (kk > 0 || !first) ? 1u : 0u);
          umma_commit(&empty[st]);
          if (last) umma_commit(&acc_done[b]);
          if (kWaitProfileDs) pc[2] += tick() - w1;
          ++t;
        } while (!last);
        if (!last) break;  // a wait gave up
      }
      if (kWaitProfileDs)
        for (int k = 0; k < 3; ++k) atomicAdd(&P.status->wait_cycles[10 + k], (unsigned long long)pc[k]);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue
    const int q = warp - 4;  // tensor memory lane quadrant
    const int r = q * 32 + lane, seg = r >> 6, rr = r & 63;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    int it_local = 0;
    for (int id = blockIdx.x; id < P.nitems && !*abort_flag; id += gridDim.x, ++it_local) {
      const int b = it_local & 1;
      const long long a0 = tick();
      if (!wait_warp(&acc_done[b], (it_local >> 1) & 1, 23)) break;
      const long long a1 = tick();
      if (kWaitProfileDs) pc[0] += a1 - a0;
      tc_fence_after();
      const Item it = decode_item_kv(g, id, P.kv_lo, P.kv_n);
      const bool valid = it.valid[seg];
      const int tok = it.I[seg] * kBlock + rr;
      __nv_bfloat16* orow = P.dq + ((size_t)tok * g.Hq + it.h[seg]) * 128;
      if (P.rope) {
        // dQ of the un-rotated queries: y_i = c (x_i cos phi + x_{i+64} sin phi),
        // y_{i+64} = c (x_{i+64} cos phi - x_i sin phi), phi = tok theta_i
        // reduced to a turn as the RoPE kernel reduces it
        const float kTurnToRad = 1.4629180792671596e-09f;  // 2 pi / 2^32
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 32) {
          uint32_t lo[32], hi[32];
          tmem_ld32(tbase + (uint32_t)(b * 128) + lane_off + c0, lo);
          tmem_ld32(tbase + (uint32_t)(b * 128) + lane_off + c0 + 64, hi);
          tmem_ld_wait();
          if (valid) {
            uint32_t ql[16], qh[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              float yl[2], yh[2];
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const uint64_t frac = (uint64_t)tok * P.rope_turn[c0 + 2 * k + e];  // modulo 2^64
                const float phi = (float)(int32_t)(uint32_t)(frac >> 32) * kTurnToRad;
                // phi is already in [-pi, pi): the hardware sine and cosine
                // (absolute error below 4e-7 there) are far inside the bf16
                // rounding of the result
                const float sn = __sinf(phi), cs = __cosf(phi);
                const float x = __uint_as_float(lo[2 * k + e]) * P.scale;
                const float y = __uint_as_float(hi[2 * k + e]) * P.scale;
                yl[e] = P.rope_mscale * (x * cs + y * sn);
                yh[e] = P.rope_mscale * (y * cs - x * sn);
              }
              ql[k] = pack_bf16(yl[0], yl[1]);
              qh[k] = pack_bf16(yh[0], yh[1]);
            }
            uint4* dl = reinterpret_cast<uint4*>(orow + c0);
            uint4* dh = reinterpret_cast<uint4*>(orow + c0 + 64);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              dl[k] = make_uint4(ql[4 * k], ql[4 * k + 1], ql[4 * k + 2], ql[4 * k + 3]);
              dh[k] = make_uint4(qh[4 * k], qh[4 * k + 1], qh[4 * k + 2], qh[4 * k + 3]);
            }
          }
        }
      } else {
        for (int c0 = 0; c0 < 128; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(tbase + (uint32_t)(b * 128) + lane_off + c0, o);
          tmem_ld_wait();
          if (valid) {
            uint32_t q16[16];
#pragma unroll
            for (int k = 0; k < 16; ++k)
              q16[k] = pack_bf16(__uint_as_float(o[2 * k]) * P.scale, __uint_as_float(o[2 * k + 1]) * P.scale);
            uint4* dst = reinterpret_cast<uint4*>(orow + c0);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              dst[k] = make_uint4(q16[4 * k], q16[4 * k + 1], q16[4 * k + 2], q16[4 * k + 3]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_free[b]);
      if (kWaitProfileDs) pc[1] += tick() - a1;
    }
    if (kWaitProfileDs && lane == 0 && warp == 4)
      for (int k = 0; k < 2; ++k) atomicAdd(&P.status->wait_cycles[20 + k], (unsigned long long)pc[k]);
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tbase, 256);
  if (kWaitProfileDs && threadIdx.x == 0) atomicAdd(&P.status->wait_cycles[kWaitSites - 1], (unsigned long long)(clock64() - k0));
}

}  // namespace

cudaError_t launch_ds_plan(const AttnGeom& g, const PrepPtrs& pp, const DsPlan& d, cudaStream_t s) {
  // any non-zero value means the tiles fit; the plan clears it otherwise
  cudaError_t e = cudaMemsetAsync(d.ok, 1, 4, s);
  if (e != cudaSuccess) return e;
  ds_plan_kernel<<<g.Hq, 1024, 0, s>>>(g, pp.inS, pp.vcnt, d);
  return cudaGetLastError();
}

cudaError_t launch_dq_stored(const vs_params& p, const AttnGeom& g, const PrepPtrs& pp, const void* K,
                             const DsPlan& d, void* dQ, DevStatus* st, int kv_lo, int kv_n, cudaStream_t s) {
  CUtensorMap mDS, mK, mKp;
  if (kv_lo < 0 || kv_n < 1 || kv_lo + kv_n > g.Hkv) return cudaErrorInvalidValue;
  if (!make_map_rows(&mDS, d.ds, ((long long)d.hpp * d.cap + 1) * 64, 64) ||
      !make_map_heads(&mK, K, g.L, g.Hkv, 128) || !make_map_rows(&mKp, pp.Kp, (long long)g.nvg * g.L, 128))
    return cudaErrorInvalidValue;
  DqsParams P;
  P.g = g;
  P.inS = pp.inS;
  P.vlist = pp.vlist;
  P.vcnt = pp.vcnt;
  P.base_s = d.base_s;
  P.base_v = d.base_v;
  P.ok = d.ok;
  P.dq = static_cast<__nv_bfloat16*>(dQ);
  P.zero_blk = d.zero_blk;
  P.kv_lo = kv_lo;
  P.kv_n = kv_n;
  P.nitems = g.nitems / g.Hkv * kv_n;
  P.scale = default_scale(p);
  P.status = st;
  P.rope = p.rope_mode == 1 ? 1 : 0;
  P.rope_mscale = 1.f;
  for (int i = 0; i < 64; ++i) P.rope_turn[i] = 0;
  if (P.rope) {
    RopeArgs ra;
    rope_fill(p, ra);
    P.rope_mscale = ra.mscale;
    for (int i = 0; i < 64; ++i) P.rope_turn[i] = ra.turn[i];
  }
  const size_t smem = kQsSmem + 1024;
  cudaError_t e = cudaFuncSetAttribute(dq_stored_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int dev = 0, nsm = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  const int grid = P.nitems < nsm ? P.nitems : nsm;
  dq_stored_kernel<<<grid, kQsThreads, smem, s>>>(mDS, mK, mKp, P);
  return cudaGetLastError();
}

}  // namespace vs
