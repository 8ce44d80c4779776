// Query-major block-sparse causal attention on the active VS entries
// (tcgen05): the forward pass, and the dQ part of the backward pass.
//
// MTraining review, section "分布式稀疏索引近似" (each worker computes only the
// active regions of its sub-matrix derived from the vertical and slash
// indices) with the online softmax across key blocks of the ring-attention
// page (section 2.1).  For each 128-row tile the kernel walks the tile's
// active key sources (64-key slash blocks and 64-entry vertical chunks, two
// per step):
//   forward:  S = Q K^T into TMEM, mask, online max / sum, P (bf16) written
//             back into TMEM, O += P V with the A operand read from TMEM;
//   dQ:       S = Q K^T and dP = dO V^T into TMEM, P = exp(scale S - LSE),
//             dS = P (dP - D) (bf16) into TMEM, dQ += dS K.
//
// Persistent CTAs (one per SM), 8 warps:
//   warp 0     producer: enumerates the tile's key sources, builds per-column
//              masks, issues TMA loads of Q (and dO) per row tile and of K
//   warp 3     second producer: the same enumeration, TMA loads of V
//   warp 1     MMA issuer (one thread)
//   warp 2     owns the TMEM allocation
//   warps 4-11 two softmax / dS warpgroups: group g handles the key columns
//              of source slot g (64 keys) for all 128 rows; thread r of a
//              group owns row r (TMEM lane r)
// K and V sit in separate rings so each is released as soon as its last
// reader is done: forward K after S (3 deep), V after O += P V (2 deep); dQ
// V after dP (2 deep), K after dQ += dS K (3 deep).  Per-tile metadata has
// its own ring, released by the softmax warps once they copied it.
// TMEM columns: S double buffer [0,128) and [128,256); P or dS of source
// slot g are written packed (bf16) over the first 32 columns of that slot's
// scores ([64 g, 64 g + 32) of the S buffer).  Forward: two accumulators,
// O_A at [256, 256+d) for slot 0 and O_B at [384, 384+d) for slot 1, each
// with its own running max and sum (independent online softmax per group),
// combined per row in the epilogue.  dQ: dP at [256, 384), dQ at [384, 384+d).
// The forward rescales lazily: only when a group's row maximum grows by more
// than 8 (log2 units) is its accumulator multiplied down; otherwise
// exponentials are taken against the stale maximum, which is exact after the
// final normalisation.
// tcgen05.ld/st are warp-collective: every branch around them is warp-uniform.
#include "attn_common.cuh"
#include "ptx.cuh"

namespace vs {
namespace {

constexpr int kThreads = 384;
constexpr float kNegInf = -__builtin_huge_valf();
constexpr float kRescaleThreshold = 8.0f;

struct TileMeta {
  uint32_t mask[2][4];  // per segment, columns 0..127 active (before the causal rule)
  int32_t diag[2];      // per segment: column offset of the diagonal source, or -1
  int32_t nsrc;         // 1 or 2 sources of 64 keys
  int32_t first, last;  // first / last tile of the row tile
  int32_t qslot;
  uint32_t mma;         // the MMA thread's copy: nsrc | first << 2 | last << 3 | qslot << 4
};

struct QmParams {
  AttnGeom g;
  const uint32_t* inS;
  const uint32_t* vlist;
  const int32_t* vcnt;
  __nv_bfloat16* out;  // O (forward) or dQ, rows of global tokens
  float* lse;          // forward: written; dQ: read ([Hq][L_glob])
  const float* Dsum;   // dQ: rowsum(dO * O) ([Hq][L_glob])
  float scale_log2;
  float scale;
  DevStatus* status;
  // ring steps: kAcc* mode and the fp32 state carried between steps, in
  // local rows: the output [L][Hq][D] (forward: normalised O; dQ: the sum so
  // far) and, forward only, the log2-domain log-sum-exp [Hq][L]
  int acc_mode;
  float* carry_o;
  float* carry_lse2;
  int item_lo, item_hi;  // row tiles [item_lo, item_hi) of the heaviest-first order
  int prod_item_hi;      // ring steps: the producers' bound, item_hi (item_lo in the bounded-wait test)
  const int32_t* skip_if;  // non-zero device word: the launch does nothing
};

template <int D, bool kDQ>
struct Layout {
  static constexpr int kHalves = D / 64;
  static constexpr int kRowBytes = 128 * 128;            // 128 rows x 128 bytes (one 64-wide d half)
  static constexpr int kQBytes = kHalves * kRowBytes;    // 128 rows of Q (or dO)
  static constexpr int kKBytes = kHalves * kRowBytes;    // 128 keys of K (or V)
  static constexpr int kQSlots = kDQ ? 1 : 2;            // dQ: one slot holding Q then dO
  static constexpr int kSlotBytes = kDQ ? 2 * kQBytes : kQBytes;
  static constexpr int kRK = 3;                          // K ring depth
  static constexpr int kRV = 2;                          // V ring depth
  static constexpr int kQ = 0;
  static constexpr int kKRing = 2 * kQBytes;
  static constexpr int kVRing = kKRing + kRK * kKBytes;
  static constexpr int kMeta = kVRing + kRV * kKBytes;
  static constexpr int kBars = (kMeta + kRK * (int)sizeof(TileMeta) + 15) / 16 * 16;  // mbarriers: 8-byte aligned
  // q_full[2], q_empty[2], k_full[RK], k_empty[RK], v_full[RV], v_empty[RV], meta_free[RK],
  // s_full[2], p_ready[2], pv_done, o_free, dp_full, dp_free, ep_a, ep_b, acc_done
  static constexpr int kNumBars = 2 + 2 + 3 * kRK + 2 * kRV + 2 + 2 + 1 + 1 + 1 + 1 + 2 + 1;
  static constexpr int kMisc = kBars + kNumBars * 8;      // tmem slot, abort flag
  static constexpr int kWaitCyc = kMisc + 64;             // per-site wait cycle counters
  static constexpr int kXchg = kWaitCyc + kWaitSites * 8; // epilogue row exchange: 128 x 2 floats
  static constexpr int kSmemEnd = kXchg + 128 * 2 * 4;
  static_assert(kBars % 8 == 0 && kMisc % 8 == 0 && kWaitCyc % 8 == 0, "mbarriers and counters need 8-byte alignment");
};

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ bool band_kept(const uint32_t* bm, int B) { return (bm[B >> 5] >> (B & 31)) & 1u; }

// Masking mode of one 64-key source for one segment's rows (warp-uniform):
// inactive, fully active, the causal diagonal block, or per-column bits.
enum : int { kSrcOff = 0, kSrcFull = 1, kSrcDiag = 2, kSrcBits = 3 };
__device__ __forceinline__ int src_mode(uint32_t w0, uint32_t w1, bool is_diag) {
  if ((w0 | w1) == 0u) return kSrcOff;
  if (is_diag) return kSrcDiag;
  if ((w0 & w1) == 0xffffffffu) return kSrcFull;
  return kSrcBits;
}
// Active columns of a 64-key source for row rr of the segment, as a 64-bit mask.
__device__ __forceinline__ uint64_t active_bits(int mode, uint32_t w0, uint32_t w1, int rr, int strict) {
  if (mode == kSrcOff) return 0ull;
  if (mode == kSrcFull) return ~0ull;
  if (mode == kSrcDiag) return diag_bits(rr, strict);
  return (uint64_t)w0 | ((uint64_t)w1 << 32);
}
// Multiply one row of the TMEM accumulator by f (warp-collective; kept out of
// line because it runs rarely and would otherwise bloat the softmax loop).
template <int D>
__device__ __noinline__ void rescale_acc_row(uint32_t taddr, float f) {
  for (int c0 = 0; c0 < D; c0 += 16) {
    uint32_t o[16];
    tmem_ld16(taddr + c0, o);
    tmem_ld_wait();
#pragma unroll
    for (int k = 0; k < 16; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * f);
    tmem_st16(taddr + c0, o);
  }
  tmem_st_wait();
}

template <int D, bool kDQ, bool kRing>
__global__ void __launch_bounds__(kThreads, 1)
    attn_qmajor_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mdO,
                       const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mV,
                       const __grid_constant__ CUtensorMap mKp, const __grid_constant__ CUtensorMap mVp,
                       const QmParams P) {
  using Ly = Layout<D, kDQ>;
  if (P.skip_if != nullptr && *P.skip_if != 0) return;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Ly::kBars);
  uint64_t* q_full = bars;
  uint64_t* q_empty = bars + 2;
  uint64_t* k_full = bars + 4;
  uint64_t* k_empty = k_full + Ly::kRK;
  uint64_t* v_full = k_empty + Ly::kRK;
  uint64_t* v_empty = v_full + Ly::kRV;
  uint64_t* meta_free = v_empty + Ly::kRV;
  uint64_t* s_full = meta_free + Ly::kRK;
  uint64_t* p_ready = s_full + 2;     // P (forward) or dS (dQ) written to TMEM
  uint64_t* pv_done = p_ready + 2;    // O += P V (forward) or dQ += dS K landed
  uint64_t* o_free = pv_done + 1;     // epilogue finished reading the accumulator
  uint64_t* dp_full = o_free + 1;     // dQ: dP landed
  uint64_t* dp_free = dp_full + 1;    // dQ: dP read by every row
  uint64_t* ep_a = dp_free + 1;       // forward epilogue: group 1 posted (m, l) of its rows
  uint64_t* ep_b = ep_a + 1;          // forward epilogue: group 0 posted the combination factors
  uint64_t* acc_done = ep_b + 1;      // a row tile's last accumulate landed (once per row tile)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + Ly::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + Ly::kMisc + 4);
  unsigned long long* wcyc = reinterpret_cast<unsigned long long*>(sm + Ly::kWaitCyc);
  const long long kernel_t0 = clock64();
  TileMeta* metas = reinterpret_cast<TileMeta*>(sm + Ly::kMeta);
  const AttnGeom& g = P.g;
  constexpr uint32_t kAccCol = kDQ ? 384 : 256;  // O_A or dQ (O_B at 384)
  constexpr uint32_t kDPCol = 256;               // dQ: dP

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&p_ready[i], 8);  // one arrival per softmax warp
    }
    for (int i = 0; i < Ly::kRK; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&meta_free[i], 8);
    }
    for (int i = 0; i < Ly::kRV; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    mbar_init(pv_done, 1);
    mbar_init(acc_done, 1);
    mbar_init(o_free, 8);
    mbar_init(ep_a, 4);
    mbar_init(ep_b, 4);
    mbar_init(dp_full, 1);
    mbar_init(dp_free, 8);
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

  long long wl[20] = {};  // profiling (light mode): this thread's wait cycles of sites < 20
  // A phase that is already complete costs one probe and no other shared
  // memory access: each shared memory access of the MMA thread waits behind
  // its tcgen05.mma in flight, so the abort flag is read only once the first
  // probe has failed.
  auto wait = [&](uint64_t* bar, uint32_t parity, int where) -> bool {
    const long long w0 = (kWaitProfileQm || kSmProfileQm) ? clock64() : 0;
    bool ok = mbar_try_wait(bar, parity);
    if (!ok) {
      if (*abort_flag) return false;
      // the bounded poll inline (this kernel's time follows its code shape:
      // the shared helper call measured slower here)
      const long long c0 = clock64();
      for (uint32_t i = 0; i < (1u << 26) && !ok; ++i) {
        ok = mbar_try_wait(bar, parity);
        if (!ok && clock64() - c0 > (long long)(kWaitLimitNs * 21 / 10)) break;
      }
    }
    if (kWaitProfileQm && (threadIdx.x & 31) == 0)
      atomicAdd(&wcyc[where & (kWaitSites - 1)], (unsigned long long)(clock64() - w0));
    if (kSmProfileQm && where < 20) wl[where] += clock64() - w0;
    if (ok) return true;
    *abort_flag = 1;
    report_timeout(P.status, (kDQ ? kTagDq : kTagForward) * 100 + where);
    return false;
  };
  // the same, agreed across the warp (callers then issue warp-collective
  // tcgen05 loads/stores, which every lane must execute together)
  auto wait_warp = [&](uint64_t* bar, uint32_t parity, int where) -> bool {
    return __all_sync(0xffffffffu, wait(bar, parity, where));
  };

  // ------------------------------------------------------------ producers
  // warp 0 (kprod): Q (+ dO) per row tile, per-tile metadata, K per source;
  // warp 3: V per source.  Both walk the same source enumeration.
  auto produce = [&](const bool kprod) {
    const long long prod0 = (kWaitProfileQm || kSmProfileQm) ? clock64() : 0;
    const int W = g.bs / kBlock;
    int t = 0, it_local = 0;
    if (lane == 0) {
      if (kprod) {
        tma_prefetch_desc(&mQ);
        tma_prefetch_desc(&mK);
        tma_prefetch_desc(&mKp);
        if (kDQ) tma_prefetch_desc(&mdO);
      } else {
        tma_prefetch_desc(&mV);
        tma_prefetch_desc(&mVp);
      }
    }
    for (int id = P.item_lo + (int)blockIdx.x; id < (kRing ? P.prod_item_hi : P.item_hi) && !*abort_flag;
         id += gridDim.x, ++it_local) {
      const Item it = decode_item(g, id);
      const int qslot = it_local % Ly::kQSlots;
      const uint32_t* bm0 = P.inS + (size_t)it.h[0] * g.nw;
      const uint32_t* bm1 = P.inS + (size_t)it.h[1] * g.nw;
      if (kprod && lane == 0) {
        if (wait(&q_empty[qslot], ((it_local / Ly::kQSlots) & 1) ^ 1, 1)) {
          mbar_arrive_expect_tx(&q_full[qslot], Ly::kSlotBytes);
          uint8_t* q = sm + Ly::kQ + qslot * Ly::kSlotBytes;
          for (int s = 0; s < 2; ++s)
            for (int hf = 0; hf < Ly::kHalves; ++hf) {
              tma_load_3d(q + hf * Ly::kRowBytes + s * 8192, &mQ, &q_full[qslot], hf * 64, it.h[s],
                          it.I[s] * kBlock);
              if (kDQ)
                tma_load_3d(q + Ly::kQBytes + hf * Ly::kRowBytes + s * 8192, &mdO, &q_full[qslot], hf * 64,
                            it.h[s], it.I[s] * kBlock);
            }
        }
      }
      __syncwarp();
      const int Itop = it.valid[1] ? max(it.I[0], it.I[1]) : it.I[0];

      // a segment's key block kb is an active slash source when kb <= I_s
      // and its band is kept (band 0, the diagonal tile, always is)
      auto slash_active = [&](int s, int kb) -> bool {
        if (!it.valid[s] || kb < 0 || kb > it.I[s]) return false;
        const int B = it.I[s] / W - kb / W;
        return B == 0 || band_kept(s ? bm1 : bm0, B);
      };
      // Kept-band words of the two segments for bands 32 w .. 32 w + 31 up to
      // the diagonal band Iw (band 0 forced); head-paired tiles only, where
      // both segments share the query block.
      const int Iw = it.I[0] / W;
      auto band_words = [&](int w, uint32_t* u0, uint32_t* u1) {
        *u0 = *u1 = 0u;
        if (w * 32 > Iw) return;
        uint32_t a = bm0[w], b = bm1[w];
        const int top = Iw - w * 32;
        if (top < 31) {
          a &= (2u << top) - 1u;
          b &= (2u << top) - 1u;
        }
        if (w == 0) {
          a |= 1u;
          b |= 1u;
        }
        *u0 = a;
        *u1 = b;
      };
      // ---- count the sources first so the final tile can be flagged
      int nslash = 0;
      if (g.pair_heads) {
        // band B >= 1 covers W key blocks, band 0 the blocks Iw W .. I
        int cnt = 0;
        for (int w0 = 0; w0 * 32 <= Iw; w0 += 32) {
          uint32_t u0, u1;
          band_words(w0 + lane, &u0, &u1);
          cnt += __popc((u0 | u1) & (w0 + lane == 0 ? ~1u : ~0u));
        }
        nslash = __reduce_add_sync(0xffffffffu, cnt) * W + (it.I[0] - Iw * W + 1);
      } else {
        for (int kb0 = Itop; kb0 >= 0; kb0 -= 32) {
          const int kb = kb0 - lane;
          const bool a = slash_active(0, kb) || slash_active(1, kb);
          nslash += __popc(__ballot_sync(0xffffffffu, a));
        }
      }
      const int nv = P.vcnt[(size_t)it.vg * (g.nb + 1) + Itop];
      const int nchunks = (nv + 63) / 64;
      const int total_src = nslash + nchunks;

      // pending sources of the tile being assembled
      int nsrc = 0, done_src = 0;
      int src_kind[2] = {0, 0};  // 0 slash key block, 1 vertical chunk
      int src_arg[2] = {0, 0};
      uint32_t smask[2][4];
      int sdiag[2];
      bool first = true;
      auto reset_masks = [&]() {
        for (int s = 0; s < 2; ++s) {
          for (int w = 0; w < 4; ++w) smask[s][w] = 0;
          sdiag[s] = -1;
        }
      };
      auto emit = [&]() {
        done_src += nsrc;
        const bool last = done_src == total_src;
        bool ok = true;
        if (kprod) {
          const int sk = t % Ly::kRK;
          if (lane == 0)
            ok = wait(&k_empty[sk], ((t / Ly::kRK) & 1) ^ 1, 2) && wait(&meta_free[sk], ((t / Ly::kRK) & 1) ^ 1, 3);
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (ok && lane == 0) {
            TileMeta& m = metas[sk];
            for (int s = 0; s < 2; ++s) {
              for (int w = 0; w < 4; ++w) m.mask[s][w] = smask[s][w];
              m.diag[s] = sdiag[s];
            }
            m.nsrc = nsrc;
            m.first = first ? 1 : 0;
            m.last = last ? 1 : 0;
            m.qslot = qslot;
            m.mma = (uint32_t)nsrc | (first ? 4u : 0u) | (last ? 8u : 0u) | ((uint32_t)qslot << 4);
            uint8_t* kst = sm + Ly::kKRing + sk * Ly::kKBytes;
            mbar_arrive_expect_tx(&k_full[sk], nsrc * Ly::kHalves * 8192);
            for (int j = 0; j < nsrc; ++j)
              for (int hf = 0; hf < Ly::kHalves; ++hf) {
                uint8_t* kd = kst + hf * Ly::kRowBytes + j * 8192;
                if (src_kind[j] == 0)
                  tma_load_3d(kd, &mK, &k_full[sk], hf * 64, it.g, src_arg[j] * kBlock);
                else
                  tma_load_2d(kd, &mKp, &k_full[sk], hf * 64, it.vg * g.L + src_arg[j] * 64);
              }
          }
        } else {
          const int sv = t % Ly::kRV;
          if (lane == 0) ok = wait(&v_empty[sv], ((t / Ly::kRV) & 1) ^ 1, 4);
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (ok && lane == 0) {
            uint8_t* vst = sm + Ly::kVRing + sv * Ly::kKBytes;
            mbar_arrive_expect_tx(&v_full[sv], nsrc * Ly::kHalves * 8192);
            for (int j = 0; j < nsrc; ++j)
              for (int hf = 0; hf < Ly::kHalves; ++hf) {
                uint8_t* vd = vst + hf * Ly::kRowBytes + j * 8192;
                if (src_kind[j] == 0)
                  tma_load_3d(vd, &mV, &v_full[sv], hf * 64, it.g, src_arg[j] * kBlock);
                else
                  tma_load_2d(vd, &mVp, &v_full[sv], hf * 64, it.vg * g.L + src_arg[j] * 64);
              }
          }
        }
        __syncwarp();
        ++t;
        nsrc = 0;
        first = false;
        reset_masks();
      };
      reset_masks();

      // ---- slash sources: key blocks kb = Itop, Itop-1, ..., 0
      auto push_slash = [&](int kbs, bool on0, bool on1) {
        const int j = nsrc;
        src_kind[j] = 0;
        src_arg[j] = kbs;
        const bool on[2] = {on0, on1};
        for (int s = 0; s < 2; ++s) {
          smask[s][2 * j] = on[s] ? 0xffffffffu : 0u;
          smask[s][2 * j + 1] = on[s] ? 0xffffffffu : 0u;
          if (on[s] && kbs == it.I[s]) sdiag[s] = 64 * j;
        }
        if (++nsrc == 2) emit();
      };
      if (g.pair_heads) {
        // walk the kept bands in ascending order (key blocks descending),
        // skipping empty bitmap words 32 at a time
        for (int w0 = 0; w0 * 32 <= Iw && !*abort_flag; w0 += 32) {
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
              const int lo = (Iw - B) * W, hi = min(it.I[0], lo + W - 1);
              for (int kbs = hi; kbs >= lo; --kbs) push_slash(kbs, (a0 >> bit) & 1u, (a1 >> bit) & 1u);
            }
          }
        }
      }
      for (int kb0 = Itop; kb0 >= 0 && !*abort_flag && !g.pair_heads; kb0 -= 32) {
        const int kb = kb0 - lane;
        const uint32_t b0 = __ballot_sync(0xffffffffu, slash_active(0, kb));
        const uint32_t b1 = __ballot_sync(0xffffffffu, slash_active(1, kb));
        uint32_t u = b0 | b1;
        while (u) {
          const int bit = __ffs(u) - 1;
          u &= u - 1;
          push_slash(kb0 - bit, (b0 >> bit) & 1u, (b1 >> bit) & 1u);
        }
      }
      // ---- vertical sources: 64-entry chunks of the union list below block Itop
      for (int c = 0; c < nchunks && !*abort_flag; ++c) {
        const int j = nsrc;
        src_kind[j] = 1;
        src_arg[j] = c;
        if (kprod) {
          for (int half = 0; half < 2; ++half) {
            const int u = c * 64 + half * 32 + lane;
            bool a[2] = {false, false};
            if (u < nv) {
              const uint32_t e = P.vlist[(size_t)it.vg * g.L + u];
              const int m = (int)(e & kVTokenMask);
              const uint32_t f = e >> kVFlagShift;
              const int kbm = m / kBlock;
              for (int s = 0; s < 2; ++s) {
                if (!it.valid[s] || !((f >> s) & 1u) || kbm >= it.I[s]) continue;
                const int B = it.I[s] / W - kbm / W;
                a[s] = B != 0 && !band_kept(s ? bm1 : bm0, B);
              }
            }
            smask[0][2 * j + half] = __ballot_sync(0xffffffffu, a[0]);
            smask[1][2 * j + half] = __ballot_sync(0xffffffffu, a[1]);
          }
        }
        if (++nsrc == 2) emit();
      }
      if (nsrc > 0) emit();
    }
    if ((kWaitProfileQm || kSmProfileQm) && lane == 0) atomicAdd(&wcyc[kprod ? 7 : 8], (unsigned long long)(clock64() - prod0));
  };

  if (warp == 0 || warp == 3) {
    produce(warp == 0);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescS64 = idesc_bf16(128, 64, false, false);
      constexpr uint32_t kIdescS128 = idesc_bf16(128, 128, false, false);
      constexpr uint32_t kIdescAcc = idesc_bf16(128, D, false, true);  // B (V or K) MN-major
      const uint32_t tAcc = tbase + kAccCol;
      int t = 0, it_local = 0;
      bool have_prev = false, ob_init = false;
      int prev_t = 0, prev_nsrc = 0, prev_first = 0, prev_item = 0;
      // O += P V (forward) or dQ += dS K (dQ) for the previous tile
      auto issue_acc = [&]() -> bool {
        if (!wait(&p_ready[prev_t & 1], (prev_t >> 1) & 1, 10)) return false;
        if (prev_first && prev_item > 0)
          if (!wait(o_free, (prev_item - 1) & 1, 11)) return false;
        const int pk = prev_t % Ly::kRK, pv = prev_t % Ly::kRV;
        if (!kDQ && !wait(&v_full[pv], (prev_t / Ly::kRV) & 1, 15)) return false;
        tc_fence_after();
        const long long a0 = kMmaProfileQm ? clock64() : 0;
        // B operand: V of the tile (forward) or K of the tile (dQ), MN-major
        const uint32_t bst = kDQ ? smem_u32(sm + Ly::kKRing + pk * Ly::kKBytes)
                                 : smem_u32(sm + Ly::kVRing + pv * Ly::kKBytes);
        const uint32_t pS = tbase + (uint32_t)((prev_t & 1) * 128);
        const uint64_t bd0 = sdesc_sw128(bst, Ly::kRowBytes, 1024);
        if (kDQ) {
          // dS of slot g sits at S-buffer columns [64 g, 64 g + 32)
          for (int kk = 0; kk < 4 * prev_nsrc; ++kk) {
            const uint64_t bd = sdesc_add(bd0, kk * 2048);
            umma_ts(tAcc, pS + (kk >> 2) * 64 + (kk & 3) * 8, bd, kIdescAcc, (kk > 0 || !prev_first) ? 1u : 0u);
          }
        } else {
          // O_A += P_0 V_0 and O_B += P_1 V_1: two independent chains, interleaved
          if (prev_first) ob_init = false;
          for (int kk = 0; kk < 4; ++kk) {
            umma_ts(tbase + 256, pS + kk * 8, sdesc_add(bd0, kk * 2048), kIdescAcc,
                    (kk > 0 || !prev_first) ? 1u : 0u);
            if (prev_nsrc == 2)
              umma_ts(tbase + 384, pS + 64 + kk * 8, sdesc_add(bd0, (kk + 4) * 2048),
                      kIdescAcc, (kk > 0 || ob_init) ? 1u : 0u);
          }
          if (prev_nsrc == 2) ob_init = true;
        }
        umma_commit(pv_done);
        if (kDQ)
          umma_commit(&k_empty[pk]);
        else
          umma_commit(&v_empty[pv]);
        if (kMmaProfileQm) atomicAdd(&wcyc[19], (unsigned long long)(clock64() - a0));
        return true;
      };
      for (int id = P.item_lo + (int)blockIdx.x; id < P.item_hi && !*abort_flag; id += gridDim.x, ++it_local) {
        bool last = false;
        do {
          const int sk = t % Ly::kRK, sv = t % Ly::kRV;
          if (!wait(&k_full[sk], (t / Ly::kRK) & 1, 12)) break;
          const long long mc0 = kSmProfileQm ? clock64() : 0;
          // one shared memory load for the fields the MMA thread uses
          const uint32_t mw = metas[sk].mma;
          const struct {
            int nsrc, first, last, qslot;
          } m = {(int)(mw & 3u), (int)((mw >> 2) & 1u), (int)((mw >> 3) & 1u), (int)(mw >> 4)};
          last = m.last != 0;
          if (m.first)
            if (!wait(&q_full[m.qslot], (it_local / Ly::kQSlots) & 1, 13)) break;
          tc_fence_after();
          if (kSmProfileQm) wl[5] += clock64() - mc0;  // metadata copy + fence (and q_full)
          const uint32_t qa = smem_u32(sm + Ly::kQ + m.qslot * Ly::kSlotBytes);
          const uint32_t kb = smem_u32(sm + Ly::kKRing + sk * Ly::kKBytes);
          const uint32_t dS = tbase + (uint32_t)((t & 1) * 128);
          const uint32_t idS = m.nsrc == 2 ? kIdescS128 : kIdescS64;
          const long long s0 = kMmaProfileQm ? clock64() : 0;
          const uint64_t qd0 = sdesc_sw128(qa, 16, 1024), kd0 = sdesc_sw128(kb, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * Ly::kRowBytes + (kk & 3) * 32;
            umma_ss(dS, sdesc_add(qd0, off), sdesc_add(kd0, off), idS, kk > 0 ? 1u : 0u);
          }
          umma_commit(&s_full[t & 1]);
          if (kMmaProfileQm) atomicAdd(&wcyc[0], (unsigned long long)(clock64() - s0));
          const long long kc0 = kSmProfileQm ? clock64() : 0;
          if (!kDQ) umma_commit(&k_empty[sk]);  // forward: K is read only by S
          if (kSmProfileQm) wl[6] += clock64() - kc0;
          if (kDQ) {
            // dP = dO V^T into the single dP buffer, once every row read the previous one
            if (t > 0 && !wait(dp_free, (t - 1) & 1, 14)) break;
            if (!wait(&v_full[sv], (t / Ly::kRV) & 1, 15)) break;
            tc_fence_after();
            const long long d0 = kMmaProfileQm ? clock64() : 0;
            const uint32_t oa = qa + Ly::kQBytes;
            const uint32_t vb = smem_u32(sm + Ly::kVRing + sv * Ly::kKBytes);
            const uint64_t od0 = sdesc_sw128(oa, 16, 1024), vd0 = sdesc_sw128(vb, 16, 1024);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk >> 2) * Ly::kRowBytes + (kk & 3) * 32;
              umma_ss(tbase + kDPCol, sdesc_add(od0, off), sdesc_add(vd0, off), idS, kk > 0 ? 1u : 0u);
            }
            umma_commit(dp_full);
            umma_commit(&v_empty[sv]);  // dQ: V is read only by dP
            if (kMmaProfileQm) atomicAdd(&wcyc[9], (unsigned long long)(clock64() - d0));
          }
          if (last) umma_commit(&q_empty[m.qslot]);
          if (kMmaProfileQm) {
            atomicAdd(&wcyc[16], 1ull);
            atomicAdd(&wcyc[17], (unsigned long long)m.nsrc);
            if (last) atomicAdd(&wcyc[18], 1ull);
          }
          if (have_prev && !issue_acc()) break;
          have_prev = true;
          prev_t = t;
          prev_nsrc = m.nsrc;
          prev_first = m.first;
          prev_item = it_local;
          // the row tile's epilogue waits for its last accumulate: issue it
          // now rather than behind the next row tile's first S
          if (last) {
            if (!issue_acc()) break;
            umma_commit(acc_done);
            have_prev = false;
          }
          ++t;
        } while (!last);  // a failed wait (timeout or abort) leaves by break
      }
      if (have_prev && !*abort_flag) issue_acc();
    }
    // lanes 1..31 wait here for the issuing lane: the block-wide barrier
    // below is warp-aligned and must see the whole warp together
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax / dS + epilogue
    const int grp = (threadIdx.x - 128) >> 7;  // source slot handled by this warpgroup
    const int r = (threadIdx.x - 128) & 127;   // row of the tile == TMEM lane
    const int seg = r >> 6, rr = r & 63;
    const uint32_t lane_off = (uint32_t)(((warp - 4) & 3) * 32) << 16;
    // forward: this group's accumulator (O_A or O_B); dQ: its half of the dQ columns
    const uint32_t tAcc = kDQ ? tbase + kAccCol + lane_off + grp * (D / 2) : tbase + 256 + 128 * grp + lane_off;
    float* xch = reinterpret_cast<float*>(sm + Ly::kXchg);
    long long pw = 0, pk_ = 0, pe = 0;  // profiling: wait / work / epilogue cycles of this warp
    int t = 0, it_local = 0;
    for (int id = P.item_lo + (int)blockIdx.x; id < P.item_hi && !*abort_flag; id += gridDim.x, ++it_local) {
      const Item it = decode_item(g, id);
      const int tok = it.I[seg] * kBlock + rr;
      const int h = it.h[seg];
      // (a VS_DEBUG build checks the row's global position before any access)
      const bool valid =
          it.valid[seg] && VS_BOUNDS(h < g.Hq && (kRing ? g.tq(tok) : tok) < (kRing ? g.L_glob : g.L) &&
                                         (!kRing || tok < g.L),
                                     P.status, (kDQ ? kTagDq : kTagForward) * 100 + 90);
      float m_ref = kNegInf, l = 0.f;
      float lse2 = 0.f, Dr = 0.f;
      // global token of this row (a ring step views one shard of the layout)
      const int gtok = kRing ? g.tq(tok) : tok;
      const size_t grow = (size_t)h * (kRing ? g.L_glob : g.L) + gtok;
      if (kDQ && valid) {
        lse2 = P.lse[grow] * 1.4426950408889634f;
        Dr = P.Dsum[grow];
      }
      bool last = false;
      do {
        const long long q0 = kSmProfileQm ? clock64() : 0;
        const int sk = t % Ly::kRK;
        if (!wait_warp(&k_full[sk], (t / Ly::kRK) & 1, 20)) break;
        // masking mode of this group's source for this row's segment (warp-uniform)
        const uint32_t mw0 = metas[sk].mask[seg][2 * grp], mw1 = metas[sk].mask[seg][2 * grp + 1];
        const int md = src_mode(mw0, mw1, metas[sk].diag[seg] == 64 * grp);
        last = metas[sk].last != 0;
        __syncwarp();
        if (lane == 0) mbar_arrive(&meta_free[sk]);
        if (!wait_warp(&s_full[t & 1], (t >> 1) & 1, 21)) break;
        const long long q1 = kSmProfileQm ? clock64() : 0;
        if (kSmProfileQm) pw += q1 - q0;
        tc_fence_after();
        const uint32_t tS = tbase + (uint32_t)((t & 1) * 128) + lane_off + 64 * grp;  // this slot's scores
        const float c2 = P.scale_log2;
        const long long ph0 = clock64();
        long long ph_rescale = 0;
        uint32_t pk[32];
        if (kDQ) {
          // ---- dS = P (dP - D), P = exp2(scale_log2 S - lse2) on active entries
          if (!wait_warp(dp_full, t & 1, 24)) break;
          tc_fence_after();
          if (md == kSrcOff) {
            // dP is released as soon as it has been read: the next tile's
            // dP = dO V^T then overlaps this tile's arithmetic
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dp_free);
#pragma unroll
            for (int k = 0; k < 32; ++k) pk[k] = 0u;
          } else {
            uint32_t sv[64], dv[64];
            tmem_ld64(tS, sv);
            tmem_ld64(tbase + kDPCol + lane_off + 64 * grp, dv);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dp_free);
            if (md == kSrcFull) {
              const uint64_t cc = f2pack(c2, c2), ll = f2pack(-lse2, -lse2);
#pragma unroll
              for (int k = 0; k < 32; ++k) {
                float x0, x1, t0, t1;
                ffma2(x0, x1, __uint_as_float(sv[2 * k]), __uint_as_float(sv[2 * k + 1]), cc, ll);
                const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
                fadd2(t0, t1, __uint_as_float(dv[2 * k]), __uint_as_float(dv[2 * k + 1]), -Dr, -Dr);
                fmul2(t0, t1, t0, t1, p0, p1);
                pk[k] = pack_bf16(t0, t1);
              }
            } else {
              const uint64_t act = active_bits(md, mw0, mw1, rr, kRing ? g.strict_diag : 0);
#pragma unroll
              for (int k = 0; k < 32; ++k) {
                const int c = 2 * k;
                const float p0 = ((act >> c) & 1ull) ? fast_exp2(fmaf(__uint_as_float(sv[c]), c2, -lse2)) : 0.f;
                const float p1 =
                    ((act >> (c + 1)) & 1ull) ? fast_exp2(fmaf(__uint_as_float(sv[c + 1]), c2, -lse2)) : 0.f;
                pk[k] = pack_bf16(p0 * (__uint_as_float(dv[c]) - Dr), p1 * (__uint_as_float(dv[c + 1]) - Dr));
              }
            }
          }
        } else {
          uint32_t v[64];
          uint64_t act;
          float mraw = kNegInf;
          if (md != kSrcOff) {
            tmem_ld64(tS, v);
            tmem_ld_wait();
            if (md != kSrcFull) {
              // masked entries become -inf in place, so neither pass needs the mask
              act = active_bits(md, mw0, mw1, rr, kRing ? g.strict_diag : 0);
#pragma unroll
              for (int c = 0; c < 64; ++c)
                if (!((act >> c) & 1ull)) v[c] = __float_as_uint(kNegInf);
            }
            mraw = row_max64(v);
          }
          if (kWaitProfileQm && lane == 0) atomicAdd(&wcyc[26], (unsigned long long)(clock64() - ph0));
          const float m_new = (mraw == kNegInf) ? m_ref : fmaxf(m_ref, mraw * c2);
          // Rows whose maximum grew by more than the threshold rescale this
          // group's accumulator after the previous PV landed.  The TMEM
          // loads/stores are warp-collective, so the whole warp takes the
          // branch when any row needs it (factor 1 for the others).
          const bool need = m_ref != kNegInf && m_new > m_ref + kRescaleThreshold;
          if (__any_sync(0xffffffffu, need)) {
            ph_rescale = clock64();
            if (kWaitProfileQm && lane == 0) atomicAdd(&wcyc[29], 1ull << 40);  // count in the high bits
            if (!wait_warp(pv_done, (t - 1) & 1, 22)) break;
            tc_fence_after();
            const float f = need ? fast_exp2(m_ref - m_new) : 1.0f;
            rescale_acc_row<D>(tAcc, f);
            if (need) {
              l *= f;
              m_ref = m_new;
            }
            ph_rescale = clock64() - ph_rescale;
            if (kWaitProfileQm && lane == 0) atomicAdd(&wcyc[29], (unsigned long long)ph_rescale);
          }
          if (m_ref == kNegInf) m_ref = m_new;
          if (md == kSrcOff) {
#pragma unroll
            for (int k = 0; k < 32; ++k) pk[k] = 0u;
          } else {
            // a row with no active key so far (only with a strict diagonal)
            // keeps m_ref = -inf: its masked scores give exp2(-inf) = 0
            const float mneg = (kRing && m_ref == kNegInf) ? 0.f : -m_ref;
            const uint64_t cc = f2pack(c2, c2), mm = f2pack(mneg, mneg);
            float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int k = 0; k < 32; ++k) {
              float x0, x1;
              ffma2(x0, x1, __uint_as_float(v[2 * k]), __uint_as_float(v[2 * k + 1]), cc, mm);
              const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
              if (k & 1)
                fadd2(ls[2], ls[3], ls[2], ls[3], p0, p1);
              else
                fadd2(ls[0], ls[1], ls[0], ls[1], p0, p1);
              pk[k] = pack_bf16(p0, p1);
            }
            l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
          }
        }
        // P (or dS) of this slot over the first 32 columns of its scores
        tmem_st32(tS, pk);
        const long long ph1 = clock64();
        tmem_st_wait();
        if (kWaitProfileQm && lane == 0) {
          atomicAdd(&wcyc[27], (unsigned long long)(ph1 - ph0 - ph_rescale));
          atomicAdd(&wcyc[28], (unsigned long long)(clock64() - ph1));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_ready[t & 1]);
        if (kSmProfileQm) pk_ += clock64() - q1;
        if (last) {
          const long long pe0 = clock64();
          // The accumulator is complete once the row tile's last accumulate
          // landed.  pv_done cannot say so: at this point the accumulates of
          // tiles t-1 and t may each have landed or not, three phases apart,
          // and a parity wait tells only two apart.  acc_done completes once
          // per row tile, and the next one needs this warp's next p_ready.
          if (!wait_warp(acc_done, it_local & 1, 23)) break;
          tc_fence_after();
          __nv_bfloat16* orow = P.out + ((size_t)gtok * g.Hq + h) * D;
          // ring steps carry an fp32 row of local token tok between steps
          float* crow = kRing ? P.carry_o + ((size_t)tok * g.Hq + h) * D + grp * (D / 2) : nullptr;
          const bool final_out = !kRing || P.acc_mode == kAccPlain || P.acc_mode == kAccLast;
          const bool read_carry = kRing && (P.acc_mode == kAccMid || P.acc_mode == kAccLast);
          if (kDQ) {
            // this group's half of the dQ columns (a ring step adds the
            // carried sum of the earlier steps)
            for (int c0 = 0; c0 < D / 2; c0 += 16) {
              uint32_t o[16];
              tmem_ld16(tAcc + c0, o);
              tmem_ld_wait();
              float x[16];
#pragma unroll
              for (int k = 0; k < 16; ++k) x[k] = __uint_as_float(o[k]) * P.scale;
              if (valid && read_carry) {
                const float4* cr = reinterpret_cast<const float4*>(crow + c0);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  const float4 v4 = cr[k];
                  x[4 * k] += v4.x;
                  x[4 * k + 1] += v4.y;
                  x[4 * k + 2] += v4.z;
                  x[4 * k + 3] += v4.w;
                }
              }
              if (valid && final_out) {
                uint32_t q8[8];
                for (int k = 0; k < 8; ++k) q8[k] = pack_bf16(x[2 * k], x[2 * k + 1]);
                uint4* dst = reinterpret_cast<uint4*>(orow + grp * (D / 2) + c0);
                dst[0] = make_uint4(q8[0], q8[1], q8[2], q8[3]);
                dst[1] = make_uint4(q8[4], q8[5], q8[6], q8[7]);
              } else if (valid) {
                float4* cw = reinterpret_cast<float4*>(crow + c0);
#pragma unroll
                for (int k = 0; k < 4; ++k) cw[k] = make_float4(x[4 * k], x[4 * k + 1], x[4 * k + 2], x[4 * k + 3]);
              }
            }
          } else {
            // Combine the row's softmax states into normalised factors: the
            // two groups' accumulators (running max m, sum l each) and, for a
            // ring step after the first, the state carried from the earlier
            // steps (a normalised output and its log2-domain log-sum-exp).
            // lse2n = log2(2^lc2 + l_A 2^m_A + l_B 2^m_B); each part's factor
            // is 2^(its max - lse2n).  Group 1 posts (m, l), group 0 posts
            // its own factor and lse2n, and each side forms the rest.
            const float lc2 = (valid && read_carry) ? P.carry_lse2[(size_t)h * g.L + tok] : kNegInf;
            float ca, cb, cc = 0.f;
            if constexpr (!kRing) {
              // a plain call: group 1 posts (m, l); group 0 forms both groups'
              // normalised factors and the row's LSE and posts the factors
              if (grp == 1) {
                xch[2 * r] = m_ref;
                xch[2 * r + 1] = l;
                __syncwarp();
                if (lane == 0) mbar_arrive(ep_a);
                if (!wait_warp(ep_b, it_local & 1, 5)) break;
                ca = xch[2 * r];
                cb = xch[2 * r + 1];
              } else {
                if (!wait_warp(ep_a, it_local & 1, 6)) break;
                const float mb = xch[2 * r], lb = xch[2 * r + 1];
                const float m = fmaxf(m_ref, mb);
                const float fa = (l > 0.f) ? fast_exp2(m_ref - m) : 0.f;
                const float fb = (lb > 0.f) ? fast_exp2(mb - m) : 0.f;
                const float ltot = l * fa + lb * fb;
                const float inv = ltot > 0.f ? 1.0f / ltot : 0.f;
                ca = fa * inv;
                cb = fb * inv;
                if (valid) P.lse[grow] = ltot > 0.f ? (m + __log2f(ltot)) * 0.69314718055994531f : kNegInf;
                xch[2 * r] = ca;
                xch[2 * r + 1] = cb;
                __syncwarp();
                if (lane == 0) mbar_arrive(ep_b);
              }
            } else if (grp == 1) {
              xch[2 * r] = m_ref;
              xch[2 * r + 1] = l;
              __syncwarp();
              if (lane == 0) mbar_arrive(ep_a);
              if (!wait_warp(ep_b, it_local & 1, 5)) break;
              ca = xch[2 * r];
              const float lse2n = xch[2 * r + 1];
              cb = (l > 0.f) ? fast_exp2(m_ref - lse2n) : 0.f;
              cc = (lc2 != kNegInf) ? fast_exp2(lc2 - lse2n) : 0.f;
            } else {
              if (!wait_warp(ep_a, it_local & 1, 6)) break;
              const float mb = xch[2 * r], lb = xch[2 * r + 1];
              float mx = lc2;
              if (l > 0.f) mx = fmaxf(mx, m_ref);
              if (lb > 0.f) mx = fmaxf(mx, mb);
              float sum = 0.f;
              if (lc2 != kNegInf) sum += fast_exp2(lc2 - mx);
              if (l > 0.f) sum += l * fast_exp2(m_ref - mx);
              if (lb > 0.f) sum += lb * fast_exp2(mb - mx);
              const float lse2n = sum > 0.f ? mx + __log2f(sum) : kNegInf;
              ca = (l > 0.f) ? fast_exp2(m_ref - lse2n) : 0.f;
              cb = (lb > 0.f) ? fast_exp2(mb - lse2n) : 0.f;
              cc = (lc2 != kNegInf) ? fast_exp2(lc2 - lse2n) : 0.f;
              if (valid) {
                if (final_out)
                  P.lse[grow] = lse2n != kNegInf ? lse2n * 0.69314718055994531f : kNegInf;
                else
                  P.carry_lse2[(size_t)h * g.L + tok] = lse2n;
              }
              xch[2 * r] = ca;
              xch[2 * r + 1] = lse2n;
              __syncwarp();
              if (lane == 0) mbar_arrive(ep_b);
            }
            // this group's half of the output columns from both accumulators
            // (and the carried output of the earlier ring steps)
            const uint32_t tA = tbase + 256 + lane_off + grp * (D / 2), tB = tA + 128;
            for (int c0 = 0; c0 < D / 2; c0 += 16) {
              uint32_t oa[16], ob[16];
              tmem_ld16(tA + c0, oa);
              tmem_ld16(tB + c0, ob);
              tmem_ld_wait();
              float x[16];
#pragma unroll
              for (int k = 0; k < 16; ++k)
                // an accumulator with no contribution (factor 0) may hold stale data
                x[k] = ca * __uint_as_float(oa[k]) + (cb != 0.f ? cb * __uint_as_float(ob[k]) : 0.f);
              if (valid && cc != 0.f) {
                const float4* cr = reinterpret_cast<const float4*>(crow + c0);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  const float4 v4 = cr[k];
                  x[4 * k] += cc * v4.x;
                  x[4 * k + 1] += cc * v4.y;
                  x[4 * k + 2] += cc * v4.z;
                  x[4 * k + 3] += cc * v4.w;
                }
              }
              if (valid && final_out) {
                uint32_t q8[8];
                for (int k = 0; k < 8; ++k) q8[k] = pack_bf16(x[2 * k], x[2 * k + 1]);
                uint4* dst = reinterpret_cast<uint4*>(orow + grp * (D / 2) + c0);
                dst[0] = make_uint4(q8[0], q8[1], q8[2], q8[3]);
                dst[1] = make_uint4(q8[4], q8[5], q8[6], q8[7]);
              } else if (valid) {
                float4* cw = reinterpret_cast<float4*>(crow + c0);
#pragma unroll
                for (int k = 0; k < 4; ++k) cw[k] = make_float4(x[4 * k], x[4 * k + 1], x[4 * k + 2], x[4 * k + 3]);
              }
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(o_free);
          if (kWaitProfileQm && lane == 0) atomicAdd(&wcyc[30], (unsigned long long)(clock64() - pe0));
          if (kSmProfileQm) pe += clock64() - pe0;
        }
        ++t;
      } while (!last && !*abort_flag);
    }
    if (kSmProfileQm && lane == 0) {
      atomicAdd(&wcyc[21], (unsigned long long)pw);
      atomicAdd(&wcyc[27], (unsigned long long)pk_);
      atomicAdd(&wcyc[30], (unsigned long long)pe);
    }
  }
  __syncwarp();
  if (kSmProfileQm && lane == 0 && warp < 4)
    for (int k = 1; k < 20; ++k)
      if (k != 9 && wl[k]) atomicAdd(&wcyc[k], (unsigned long long)wl[k]);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tbase, 512);
  if (kMmaProfileQm && threadIdx.x < kWaitSites - 1 && wcyc[threadIdx.x])
    atomicAdd(&P.status->wait_cycles[threadIdx.x], wcyc[threadIdx.x]);
  if (kMmaProfileQm && threadIdx.x == kWaitSites - 1)
    atomicAdd(&P.status->wait_cycles[kWaitSites - 1], (unsigned long long)(clock64() - kernel_t0));
}

template <int D, bool kDQ, bool kRing>
cudaError_t launch_qmajor(const AttnGeom& g, const PrepPtrs& pp, const void* Q, const void* dO, const void* K,
                          const void* V, const QmParams& P, cudaStream_t s) {
  using Ly = Layout<D, kDQ>;
  CUtensorMap mQ, mdO, mK, mV, mKp, mVp;
  if (!make_map_heads(&mQ, Q, g.L, g.Hq, D, g.tq_mul, g.tq_add) ||
      !make_map_heads(&mdO, kDQ ? dO : Q, g.L, g.Hq, D, g.tq_mul, g.tq_add) ||
      !make_map_heads(&mK, K, g.L, g.Hkv, D, g.tk_mul, g.tk_add) ||
      !make_map_heads(&mV, V, g.L, g.Hkv, D, g.tk_mul, g.tk_add) ||
      !make_map_rows(&mKp, pp.Kp, (long long)g.nvg * g.L, D) ||
      !make_map_rows(&mVp, pp.Vp, (long long)g.nvg * g.L, D))
    return cudaErrorInvalidValue;
  const size_t smem = Ly::kSmemEnd + 1024;
  cudaError_t e =
      cudaFuncSetAttribute(attn_qmajor_kernel<D, kDQ, kRing>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int dev = 0, nsm = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  const int n = P.item_hi - P.item_lo;
  if (n <= 0) return cudaSuccess;
  const int grid = n < nsm ? n : nsm;
  attn_qmajor_kernel<D, kDQ, kRing><<<grid, kThreads, smem, s>>>(mQ, mdO, mK, mV, mKp, mVp, P);
  return cudaGetLastError();
}

}  // namespace

size_t attn_fwd_ws_bytes(const vs_params& p) {
  const AttnGeom g = make_geom(p);
  WsLayout w;
  w.take(sizeof(DevStatus));
  prep_layout(g, w);
  return w.off;
}

namespace {
// a ring step (token-strided shard views, strict diagonal or carried state)
// runs the kernel instance compiled with that support; a plain call runs
// the one without it
bool is_ring_step(const AttnGeom& g, const StepCtl& ctl) {
  return ctl.acc_mode != kAccPlain || g.strict_diag || g.tq_mul != 1 || g.tk_mul != 1 || g.tq_add != 0 ||
         g.tk_add != 0 || g.L_glob != g.L;
}

void set_step(QmParams& P, const AttnGeom& g, const StepCtl& ctl) {
  P.acc_mode = ctl.acc_mode;
  P.carry_o = ctl.carry_o;
  P.carry_lse2 = ctl.carry_lse2;
  P.item_lo = ctl.item_lo < 0 ? 0 : ctl.item_lo;
  P.item_hi = (ctl.item_hi < 0 || ctl.item_hi > g.nitems) ? g.nitems : ctl.item_hi;
  P.prod_item_hi = test_stall_requested() ? P.item_lo : P.item_hi;
  P.skip_if = ctl.skip_if;
}
}  // namespace

cudaError_t launch_fwd_core(const vs_params& p, const AttnGeom& g, const PrepPtrs& pp, const void* Q, const void* K,
                            const void* V, void* O, float* lse, DevStatus* st, const StepCtl& ctl, cudaStream_t s) {
  QmParams P;
  P.g = g;
  P.inS = pp.inS;
  P.vlist = pp.vlist;
  P.vcnt = pp.vcnt;
  P.out = static_cast<__nv_bfloat16*>(O);
  P.lse = lse;
  P.Dsum = nullptr;
  P.scale = default_scale(p);
  P.scale_log2 = P.scale * 1.4426950408889634f;
  P.status = st;
  set_step(P, g, ctl);
  if (is_ring_step(g, ctl)) {
    if (p.d == 128) return launch_qmajor<128, false, true>(g, pp, Q, nullptr, K, V, P, s);
    return launch_qmajor<64, false, true>(g, pp, Q, nullptr, K, V, P, s);
  }
  if (p.d == 128) return launch_qmajor<128, false, false>(g, pp, Q, nullptr, K, V, P, s);
  return launch_qmajor<64, false, false>(g, pp, Q, nullptr, K, V, P, s);
}

// Row tiles covering query blocks [blk_lo, blk_hi) in the heaviest-first
// numbering of decode_item (head-paired tiles: one block each; otherwise
// block pairs, so the range is widened to whole pairs).
void item_range(const AttnGeom& g, int blk_lo, int blk_hi, int* lo, int* hi) {
  if (g.pair_heads) {
    *lo = (g.nb - blk_hi) * g.items_per_row;
    *hi = (g.nb - blk_lo) * g.items_per_row;
  } else {
    const int npair = (g.nb + 1) / 2;
    const int u_lo = blk_lo / 2, u_hi = (blk_hi + 1) / 2;
    *lo = (npair - u_hi) * g.items_per_row;
    *hi = (npair - u_lo) * g.items_per_row;
  }
}

cudaError_t launch_attn_fwd(const vs_params& p, const vs_index& ix, const void* Q, const void* K, const void* V,
                            void* O, float* lse, void* ws, cudaStream_t s, int blk_lo, int blk_hi) {
  const AttnGeom g = make_geom(p);
  uint8_t* w = static_cast<uint8_t*>(ws);
  WsLayout lay;
  const size_t st_off = lay.take(sizeof(DevStatus));
  const PrepWs pw = prep_layout(g, lay);
  PrepPtrs pp;
  pp.inS = reinterpret_cast<uint32_t*>(w + pw.inS);
  pp.vlist = reinterpret_cast<uint32_t*>(w + pw.vlist);
  pp.vcnt = reinterpret_cast<int32_t*>(w + pw.vcnt);
  pp.Kp = reinterpret_cast<__nv_bfloat16*>(w + pw.Kp);
  pp.Vp = reinterpret_cast<__nv_bfloat16*>(w + pw.Vp);
  pp.vbits = pw.vbits != pw.end ? reinterpret_cast<uint32_t*>(w + pw.vbits) : nullptr;
  cudaError_t e = launch_attn_prep(g, ix, K, V, pp, s);
  if (e != cudaSuccess) return e;
  StepCtl ctl;
  if (blk_lo > 0 || blk_hi < g.nb) item_range(g, blk_lo, blk_hi, &ctl.item_lo, &ctl.item_hi);
  return launch_fwd_core(p, g, pp, Q, K, V, O, lse, reinterpret_cast<DevStatus*>(w + st_off), ctl, s);
}

cudaError_t launch_attn_dq(const vs_params& p, const AttnGeom& g, const PrepPtrs& pp, const void* Q, const void* K,
                           const void* V, const void* dO, const float* lse, const float* Dsum, void* dQ,
                           DevStatus* st, const StepCtl& ctl, cudaStream_t s) {
  QmParams P;
  P.g = g;
  P.inS = pp.inS;
  P.vlist = pp.vlist;
  P.vcnt = pp.vcnt;
  P.out = static_cast<__nv_bfloat16*>(dQ);
  P.lse = const_cast<float*>(lse);
  P.Dsum = Dsum;
  P.scale = default_scale(p);
  P.scale_log2 = P.scale * 1.4426950408889634f;
  P.status = st;
  set_step(P, g, ctl);
  if (is_ring_step(g, ctl)) {
    if (p.d == 128) return launch_qmajor<128, true, true>(g, pp, Q, dO, K, V, P, s);
    return launch_qmajor<64, true, true>(g, pp, Q, dO, K, V, P, s);
  }
  if (p.d == 128) return launch_qmajor<128, true, false>(g, pp, Q, dO, K, V, P, s);
  return launch_qmajor<64, true, false>(g, pp, Q, dO, K, V, P, s);
}

}  // namespace vs
