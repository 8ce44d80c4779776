// Sparse-index approximation, scoring stage.
//
// MTraining review, section "分布式稀疏索引近似": the last last_q query rows
// are scored against every key and the attention mass is accumulated along
// the vertical (key token) and slash (block-diagonal) directions.  Reading
// used here: s = scale * q_n . k_m over causal m <= n, p = softmax_m(s) per
// row, v[m] = sum over rows of p, S[B] = sum of p over the entries whose tile
// band n/bs - m/bs equals B (bs = 64 * stripes).
//
// Two passes over K with the same tiling (softmax needs the row maximum and
// sum before normalised probabilities can be summed per key):
//   pass 1: per (row, key chunk) running max / sum in the log2 domain
//   combine: per row global max and 1/sum
//   pass 2: p = exp2(s' - M) / l, column sums -> v, per-64-key-tile row sums
//           -> T64, then the band reduction T64 -> S.
// One CTA = one KV head x one chunk of keys x up to 256 query rows (all the
// query heads of the GQA group that fit), so each K tile is staged once in
// shared memory and reused by G * last_q rows.  QK^T runs on mma.sync
// m16n8k16 (bf16 in, fp32 accumulate); the query fragments stay in registers.
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace vs {
namespace {

constexpr int kThreads = 256;  // 8 warps x 2 m-tiles x 16 rows = 256 rows
constexpr int kRowsPerCta = 256;
constexpr float kNegInf = -__builtin_huge_valf();

__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4(uint32_t* r, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Rows per CTA are whole heads: heads_per_cta * qpad <= 256.
__host__ __device__ inline int heads_per_cta(int qpad, int G) {
  int h = kRowsPerCta / qpad;
  return h < G ? h : G;
}

template <int D, bool kPass2>
__global__ void __launch_bounds__(kThreads, 2) index_scores_kernel(const IndexArgs a) {
  constexpr int KSTR = D + 8;  // padded row (bf16): conflict-free ldmatrix
  constexpr int KSTEPS = D / 16;
  constexpr int CHUNKS16 = D / 8;  // 16-byte pieces per key row
  __shared__ __align__(16) __nv_bfloat16 ks[2][64 * KSTR];
  __shared__ float part[16][64];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const int split = blockIdx.x % a.row_splits;
  const int chunk = blockIdx.x / a.row_splits;
  const int g = blockIdx.y;
  const int hpc = heads_per_cta(a.qpad, a.G);
  const int hl0 = split * hpc;                       // first local head of this CTA
  const int nheads = min(hpc, a.G - hl0);
  const int nmt = nheads * a.qpad / 16;              // m-tiles of this CTA

  // ---- per row-slot bookkeeping: slot s = 2*j + hh (m-tile j, row half hh)
  int tok[4], rg[4], hq[4];
  bool rv[4];
  float rM[4], rInv[4];
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const int j = s >> 1, hh = s & 1;
    const int mt = warp * 2 + j;
    const int r = mt * 16 + gq + hh * 8;             // row within CTA
    const int hl = hl0 + r / a.qpad;
    const int i = r % a.qpad;
    hq[s] = g * a.G + hl;
    rv[s] = (mt < nmt) && (i < a.last_q);
    tok[s] = a.L - a.last_q + i;
    rg[s] = (mt < nmt) ? hq[s] * a.qpad + i : -1;
    rM[s] = 0.f;
    rInv[s] = 0.f;
    if (kPass2 && rv[s]) {
      const float2 st = a.rowstat[rg[s]];
      rM[s] = st.x;
      rInv[s] = st.y;
    }
  }
  // ---- query fragments (A operand, row-major 16x16 per k-step)
  uint32_t af[2][KSTEPS][4];
  const __nv_bfloat16* Qp = static_cast<const __nv_bfloat16*>(a.Q);
#pragma unroll
  for (int j = 0; j < 2; ++j) {
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk) {
      const int col = kk * 16 + tq * 2;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const int s = 2 * j + (q4 & 1);
        const int c = col + (q4 >> 1) * 8;
        uint32_t v = 0;
        if (rv[s]) v = *reinterpret_cast<const uint32_t*>(Qp + ((size_t)tok[s] * a.Hq + hq[s]) * D + c);
        af[j][kk][q4] = v;
      }
    }
  }

  const int t_begin = chunk * a.tiles_per_chunk;
  const int t_end = min(a.ntile, t_begin + a.tiles_per_chunk);
  const __nv_bfloat16* Kp = static_cast<const __nv_bfloat16*>(a.K);
  auto load_tile = [&](int t, int buf) {
    for (int c = threadIdx.x; c < 64 * CHUNKS16; c += kThreads) {
      const int r = c / CHUNKS16, p = c % CHUNKS16;
      const __nv_bfloat16* src = Kp + ((size_t)(t * 64 + r) * a.Hkv + g) * D + p * 8;
      cp_async16(smem_u32(&ks[buf][r * KSTR + p * 8]), src);
    }
    cp_async_commit();
  };

  float runM[4], runL[4];
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    runM[s] = kNegInf;
    runL[s] = 0.f;
  }

  if (t_begin < t_end) load_tile(t_begin, 0);
  for (int t = t_begin; t < t_end; ++t) {
    const int buf = (t - t_begin) & 1;
    if (t + 1 < t_end) {
      load_tile(t + 1, buf ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const bool need_mask = (t * 64 + 63) > (a.L - a.last_q);
    float rowsum[4] = {0.f, 0.f, 0.f, 0.f};
    if (warp * 2 < nmt) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float acc[2][4][4];
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[j][nt][e] = 0.f;
        const uint32_t kbase = smem_u32(&ks[buf][0]);
#pragma unroll
        for (int kk = 0; kk < KSTEPS; ++kk) {
#pragma unroll
          for (int np = 0; np < 2; ++np) {
            const int mat = lane >> 3;
            const int n = half * 32 + np * 16 + (mat >> 1) * 8 + (lane & 7);
            const int k = kk * 16 + (mat & 1) * 8;
            uint32_t b[4];
            ldsm_x4(b, kbase + (uint32_t)(n * KSTR + k) * 2u);
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              mma16816(acc[j][2 * np], af[j][kk], b[0], b[1]);
              mma16816(acc[j][2 * np + 1], af[j][kk], b[2], b[3]);
            }
          }
        }
        // ---- softmax statistics / probabilities for this 32-key half
        const int key0 = t * 64 + half * 32 + tq * 2;
        float colv[2][8];
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          const int j = s >> 1, hh = s & 1;
          float x[8];
#pragma unroll
          for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              float v = acc[j][nt][hh * 2 + e] * a.scale_log2;
              if (need_mask && key0 + nt * 8 + e > tok[s]) v = kNegInf;
              x[nt * 2 + e] = v;
            }
          }
          if (!kPass2) {
            float mx = x[0];
#pragma unroll
            for (int k = 1; k < 8; ++k) mx = fmaxf(mx, x[k]);
            const float mnew = fmaxf(runM[s], mx);
            if (mnew != kNegInf) {
              float l = runL[s] * fast_exp2(runM[s] - mnew);
#pragma unroll
              for (int k = 0; k < 8; ++k) l += fast_exp2(x[k] - mnew);
              runL[s] = l;
              runM[s] = mnew;
            }
          } else {
            float rs = 0.f;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const float p = fast_exp2(x[k] - rM[s]) * rInv[s];
              rs += p;
              if (hh == 0)
                colv[j][k] = p;
              else
                colv[j][k] += p;
            }
            rowsum[s] += rs;
          }
        }
        if (kPass2) {
          // column sums over the 16 rows of each m-tile: reduce-scatter over
          // the 8 lanes sharing a column set; lane ends with column
          // (gq>>1)*8 + 2*tq + (gq&1) of the half.
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const bool b4 = (lane >> 4) & 1, b3 = (lane >> 3) & 1, b2 = (lane >> 2) & 1;
            float k1[4], k2[2];
#pragma unroll
            for (int idx = 0; idx < 4; ++idx) {
              const float send = b4 ? colv[j][idx] : colv[j][idx + 4];
              const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
              k1[idx] = (b4 ? colv[j][idx + 4] : colv[j][idx]) + recv;
            }
#pragma unroll
            for (int idx = 0; idx < 2; ++idx) {
              const float send = b3 ? k1[idx] : k1[idx + 2];
              const float recv = __shfl_xor_sync(0xffffffffu, send, 8);
              k2[idx] = (b3 ? k1[idx + 2] : k1[idx]) + recv;
            }
            const float send = b2 ? k2[0] : k2[1];
            const float recv = __shfl_xor_sync(0xffffffffu, send, 4);
            const float fin = (b2 ? k2[1] : k2[0]) + recv;
            const int mt = warp * 2 + j;
            if (mt < nmt) part[mt][half * 32 + (gq >> 1) * 8 + tq * 2 + (gq & 1)] = fin;
          }
        }
      }
      if (kPass2) {
        // row mass of this 64-key tile (slash statistics): reduce over the 4
        // lanes of a row; lane tq ends with slot tq.
        const bool b1 = (tq >> 1) & 1, b0 = tq & 1;
        float k1[2];
#pragma unroll
        for (int idx = 0; idx < 2; ++idx) {
          const float send = b1 ? rowsum[idx] : rowsum[idx + 2];
          const float recv = __shfl_xor_sync(0xffffffffu, send, 2);
          k1[idx] = (b1 ? rowsum[idx + 2] : rowsum[idx]) + recv;
        }
        const float send = b0 ? k1[0] : k1[1];
        const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
        const float fin = (b0 ? k1[1] : k1[0]) + recv;
        const int s = tq;
        if (rv[s]) {
          const int i = tok[s] - (a.L - a.last_q);
          a.T64[((size_t)hq[s] * a.last_q + i) * a.ntile + t] = fin;
        }
      }
    }
    if (kPass2) {
      __syncthreads();
      // v[h][key] = sum over the head's m-tiles, fixed order
      const int mt_per_head = a.qpad / 16;
      for (int c = threadIdx.x; c < nheads * 64; c += kThreads) {
        const int hl = c / 64, col = c % 64;
        float sum = 0.f;
        for (int m = 0; m < mt_per_head; ++m) sum += part[hl * mt_per_head + m][col];
        a.v[(size_t)(g * a.G + hl0 + hl) * a.L + t * 64 + col] = sum;
      }
    }
    __syncthreads();
  }

  if (!kPass2) {
    // combine (max, sum) across the 4 lanes of each row
#pragma unroll
    for (int s = 0; s < 4; ++s) {
#pragma unroll
      for (int off = 1; off <= 2; off <<= 1) {
        const float om = __shfl_xor_sync(0xffffffffu, runM[s], off);
        const float ol = __shfl_xor_sync(0xffffffffu, runL[s], off);
        const float mn = fmaxf(runM[s], om);
        if (mn != kNegInf) {
          runL[s] = runL[s] * fast_exp2(runM[s] - mn) + ol * fast_exp2(om - mn);
          runM[s] = mn;
        }
      }
      if (tq == 0 && rg[s] >= 0) a.part[(size_t)chunk * a.Hq * a.qpad + rg[s]] = make_float2(runM[s], runL[s]);
    }
  }
}

__global__ void index_rowstat_kernel(const IndexArgs a) {
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  const int nrows = a.Hq * a.qpad;
  if (r >= nrows) return;
  const int i = r % a.qpad;
  if (i >= a.last_q) {
    a.rowstat[r] = make_float2(0.f, 0.f);
    return;
  }
  float M = kNegInf;
  for (int c = 0; c < a.nchunk; ++c) M = fmaxf(M, a.part[(size_t)c * nrows + r].x);
  float l = 0.f;
  for (int c = 0; c < a.nchunk; ++c) {
    const float2 p = a.part[(size_t)c * nrows + r];
    if (p.x != kNegInf) l += p.y * fast_exp2(p.x - M);
  }
  a.rowstat[r] = make_float2(M, 1.0f / l);
}

// S[h][B] = sum over index rows i and the 64-key tiles of key tile-band
// (J_i - B), J_i = n_i / bs, fixed summation order.
__global__ void index_slash_kernel(const IndexArgs a) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= a.Hq * a.nbs) return;
  const int h = idx / a.nbs, B = idx % a.nbs;
  const int W = a.bs / 64;
  float sum = 0.f;
  for (int i = 0; i < a.last_q; ++i) {
    const int J = (a.L - a.last_q + i) / a.bs;
    if (J < B) continue;
    const float* row = a.T64 + ((size_t)h * a.last_q + i) * a.ntile + (size_t)(J - B) * W;
    for (int w = 0; w < W; ++w) sum += row[w];
  }
  a.S[idx] = sum;
}

}  // namespace

void index_grid(const vs_params& p, int* tiles_per_chunk, int* nchunk, int* row_splits) {
  const int qpad = (p.last_q + 15) / 16 * 16;
  const int G = p.Hq / p.Hkv;
  const int hpc = heads_per_cta(qpad, G);
  const int rs = (G + hpc - 1) / hpc;
  const int ntile = p.L / 64;
  const int target = (2 * 152 * 2) / (p.Hkv * rs);  // about two resident waves
  int tpc = (ntile + (target > 0 ? target : 1) - 1) / (target > 0 ? target : 1);
  if (tpc < 1) tpc = 1;
  *tiles_per_chunk = tpc;
  *nchunk = (ntile + tpc - 1) / tpc;
  *row_splits = rs;
}

bool index_tc_supported(const IndexArgs& a);
cudaError_t launch_index_scores_tc(const IndexArgs& a, cudaStream_t s);

cudaError_t launch_index_scores(const IndexArgs& a, cudaStream_t s) {
  // last_q = 64: the tensor-core passes (index_tc.cu); otherwise these
  if (index_tc_supported(a)) return launch_index_scores_tc(a, s);
  dim3 grid(a.nchunk * a.row_splits, a.Hkv);
  if (a.d == 128) {
    index_scores_kernel<128, false><<<grid, kThreads, 0, s>>>(a);
  } else {
    index_scores_kernel<64, false><<<grid, kThreads, 0, s>>>(a);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int nrows = a.Hq * a.qpad;
  index_rowstat_kernel<<<(nrows + 255) / 256, 256, 0, s>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (a.d == 128) {
    index_scores_kernel<128, true><<<grid, kThreads, 0, s>>>(a);
  } else {
    index_scores_kernel<64, true><<<grid, kThreads, 0, s>>>(a);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int n = a.Hq * a.nbs;
  index_slash_kernel<<<(n + 255) / 256, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace vs
