// Preparation for the sparse attention kernels: kept-band bitmaps per head,
// the vertical union list of each tile group with per-entry membership bits
// and per-block prefix counts, and the packed K/V rows of those verticals.
#include <cudaTypedefs.h>

#include <algorithm>

#include "attn_common.cuh"

namespace vs {
namespace {

// One CTA per query head: bitmap of kept bands.
__global__ void prep_bands_kernel(AttnGeom g, const int32_t* __restrict__ s_idx, const int32_t* __restrict__ s_cnt,
                                  uint32_t* __restrict__ inS) {
  extern __shared__ uint32_t bits[];
  const int h = blockIdx.x;
  for (int w = threadIdx.x; w < g.nw; w += blockDim.x) bits[w] = 0;
  __syncthreads();
  const int n = s_cnt[h];
  for (int j = threadIdx.x; j < n; j += blockDim.x) {
    const int B = s_idx[(size_t)h * g.nbs + j];
    if (B >= 0 && B < g.nbs) atomicOr(&bits[B >> 5], 1u << (B & 31));
  }
  __syncthreads();
  for (int w = threadIdx.x; w < g.nw; w += blockDim.x) inS[(size_t)h * g.nw + w] = bits[w];
}

// One CTA per union group: bitmaps of both heads' verticals (L bits each),
// then an in-order compaction into the union list.
__global__ void __launch_bounds__(1024) prep_vunion_kernel(AttnGeom g, const int32_t* __restrict__ v_idx,
                                                           const int32_t* __restrict__ v_cnt,
                                                           uint32_t* __restrict__ vlist, int32_t* __restrict__ vcnt,
                                                           uint32_t* __restrict__ gbits) {
  extern __shared__ uint32_t sm[];
  const int nwl = g.L / 32;
  // the two heads' bitmaps: shared memory, or this pair's workspace slice
  uint32_t* bits = gbits ? gbits + (size_t)blockIdx.x * 2 * nwl : sm;
  uint32_t* b0 = bits;
  uint32_t* b1 = bits + nwl;
  __shared__ int wsum[32];
  __shared__ int carry_s;
  const int vg = blockIdx.x;
  int hs[2];
  if (g.pair_heads) {
    const int kv = vg / (g.G / 2), hp = vg % (g.G / 2);
    hs[0] = kv * g.G + 2 * hp;
    hs[1] = hs[0] + 1;
  } else {
    hs[0] = hs[1] = vg;
  }
  for (int w = threadIdx.x; w < 2 * nwl; w += blockDim.x) bits[w] = 0;
  __syncthreads();
  for (int s = 0; s < 2; ++s) {
    uint32_t* b = s ? b1 : b0;
    const int n = v_cnt[hs[s]];
    for (int j = threadIdx.x; j < n; j += blockDim.x) {
      const int m = v_idx[(size_t)hs[s] * g.L + j];
      if (m >= 0 && m < g.L) atomicOr(&b[m >> 5], 1u << (m & 31));
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) carry_s = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int base = 0; base < nwl; base += blockDim.x) {
    const int w = base + threadIdx.x;
    const uint32_t u = (w < nwl) ? (b0[w] | b1[w]) : 0u;
    const int c = __popc(u);
    int incl = c;
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int before = carry_s;
    int total = 0;
    for (int k = 0; k < (int)(blockDim.x >> 5); ++k) {
      if (k < warp) before += wsum[k];
      total += wsum[k];
    }
    int pos = before + incl - c;
    if (w < nwl) {
      if ((w & 1) == 0) vcnt[(size_t)vg * (g.nb + 1) + (w >> 1)] = pos;  // entries before block w/2
      uint32_t x = u;
      while (x) {
        const int bit = __ffs(x) - 1;
        x &= x - 1;
        const uint32_t f = ((b0[w] >> bit) & 1u) | (((b1[w] >> bit) & 1u) << 1);
        vlist[(size_t)vg * g.L + pos++] = (uint32_t)(w * 32 + bit) | (f << kVFlagShift);
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) carry_s += total;
    __syncthreads();
  }
  if (threadIdx.x == 0) vcnt[(size_t)vg * (g.nb + 1) + g.nb] = carry_s;
}

// Gather K/V rows of the union entries: one warp per row, 16 bytes per lane.
__global__ void prep_pack_kernel(AttnGeom g, const __nv_bfloat16* __restrict__ K, const __nv_bfloat16* __restrict__ V,
                                 const uint32_t* __restrict__ vlist, const int32_t* __restrict__ vcnt,
                                 __nv_bfloat16* __restrict__ Kp, __nv_bfloat16* __restrict__ Vp) {
  // blockIdx.y: the union group; its rows up to the end of the last 64-row
  // chunk, 16 bytes a thread
  const int vg = blockIdx.y;
  const int lanes_per_row = g.d / 8;
  const int cnt = vcnt[(size_t)vg * (g.nb + 1) + g.nb];
  const long long total = (long long)((cnt + 63) & ~63) * lanes_per_row;
  const int kv = g.pair_heads ? vg / (g.G / 2) : vg / g.G;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x; t < total; t += stride) {
    const int piece = (int)(t % lanes_per_row);
    const int u = (int)(t / lanes_per_row);
    const size_t dst = ((size_t)vg * g.L + u) * g.d + piece * 8;
    if (u >= cnt) {
      // zero the tail of the last 64-row chunk: masked columns there are
      // multiplied by P = 0 and must hold finite values
      *reinterpret_cast<uint4*>(Kp + dst) = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(Vp + dst) = make_uint4(0, 0, 0, 0);
      continue;
    }
    const int m = (int)(vlist[(size_t)vg * g.L + u] & kVTokenMask);
    const size_t src = ((size_t)g.tk(m) * g.Hkv + kv) * g.d + piece * 8;
    *reinterpret_cast<uint4*>(Kp + dst) = *reinterpret_cast<const uint4*>(K + src);
    *reinterpret_cast<uint4*>(Vp + dst) = *reinterpret_cast<const uint4*>(V + src);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

}  // namespace

bool make_map_heads(CUtensorMap* m, const void* base, int L, int H, int d, int tok_mul, int tok_add) {
  auto enc = encode_fn();
  if (!enc) return false;
  const char* b = static_cast<const char*>(base) + (size_t)tok_add * H * d * 2;
  base = b;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)L};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)tok_mul * H * d * 2};
  cuuint32_t box[3] = {64, 1, 64};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_strided(CUtensorMap* m, const void* base, int R, int H, int d, int S) {
  auto enc = encode_fn();
  if (!enc) return false;
  // element (x, j * H + h, c) is channel x of head h at token c * S + j
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)S * H, (cuuint64_t)R};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)S * H * d * 2};
  cuuint32_t box[3] = {64, 1, 64};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_rows(CUtensorMap* m, const void* base, long long rows, int d) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)d * 2};
  cuuint32_t box[2] = {64, 64};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_prep_bands(const AttnGeom& g, const vs_index& ix, const PrepPtrs& pp, cudaStream_t s) {
  prep_bands_kernel<<<g.Hq, 256, g.nw * 4, s>>>(g, ix.s_idx, ix.s_cnt, pp.inS);
  return cudaGetLastError();
}

cudaError_t launch_attn_prep(const AttnGeom& g, const vs_index& ix, const void* K, const void* V,
                             const PrepPtrs& pp, cudaStream_t s) {
  cudaError_t e = launch_prep_bands(g, ix, pp, s);
  if (e != cudaSuccess) return e;
  return launch_prep_verticals(g, ix, K, V, pp, s);
}

cudaError_t launch_prep_verticals(const AttnGeom& g, const vs_index& ix, const void* K, const void* V,
                                  const PrepPtrs& pp, cudaStream_t s) {
  cudaError_t e;
  const size_t bits = (size_t)2 * (g.L / 32) * 4;
  const size_t sm = pp.vbits ? 0 : bits;
  e = cudaFuncSetAttribute(prep_vunion_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  prep_vunion_kernel<<<g.nvg, 1024, sm, s>>>(g, ix.v_idx, ix.v_cnt, pp.vlist, pp.vcnt, pp.vbits);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // about eight 256-thread blocks per SM over all union groups
  const dim3 grid((unsigned)std::max(1, 152 * 8 / g.nvg), (unsigned)g.nvg);
  prep_pack_kernel<<<grid, 256, 0, s>>>(g, static_cast<const __nv_bfloat16*>(K),
                                           static_cast<const __nv_bfloat16*>(V), pp.vlist, pp.vcnt, pp.Kp, pp.Vp);
  return cudaGetLastError();
}

}  // namespace vs
