// Striped sparse ring attention, run step by step on one GPU.
//
// MTraining review, section 三/核心创新/3 "平衡稀疏环注意力" (striped layout:
// token t belongs to worker t mod W at local position t div W; one shared
// index whose slash bands are 64 x 64 tiles of the shard-local order) and the
// ring-attention page, section 2.1 (each step folds one KV block into a
// carried softmax state) and section 3.1 (striped round-robin layout).
//
// Worker r holds the queries of its shard; at step t it holds KV shard
// s = (r - t) mod W.  A step is a problem of Ls = L / W local tokens:
//   * local query row i is global token i W + r, local key row j is j W + s
//     (tensor maps with a token stride, so no shard is ever copied);
//   * slash bands are the shared index's bands, in local tiles;
//   * verticals are the kept global tokens of shard s, as local rows;
//   * the diagonal tile admits j <= i when s <= r and j < i when s > r
//     (the global causal rule m <= n).
// The forward carries (normalised O, log-sum-exp) per worker in fp32 scratch
// and folds each step in inside the attention kernel's epilogue; the last
// step writes O and LSE.  The backward uses the final LSE and
// D = rowsum(dO * O) of every query, so each step's gradients are exact
// pieces of the whole: dQ of a worker is summed over its steps in fp32
// scratch, dK / dV of a shard over all workers in fp32 sums.
// Steps run worker by worker, so a worker's carried state stays in L2.
#include "attn_common.cuh"

namespace vs {

cudaError_t launch_bwd_dsum(const void* O, const void* dO, float* Dsum, int L, int Hq, int d, cudaStream_t s);
cudaError_t launch_dkdv_core(const vs_params& p, const AttnGeom& g, const PrepPtrs& pp, const vs_index& ix,
                             const void* Q, const void* K, const void* V, const void* dO, const float* lse,
                             const float* Dsum, void* dK, void* dV, float* part_k, float* part_v, float* dk32,
                             float* dv32, DevStatus* st, const DsPlan* ds, cudaStream_t s);
size_t bwd_partials_bytes(const AttnGeom& g);

namespace {

// One CTA per (head, shard): the kept verticals of shard s as local rows,
// ascending (the global list is ascending and t -> t div W keeps the order).
__global__ void ring_shard_index_kernel(const int32_t* __restrict__ v_idx, const int32_t* __restrict__ v_cnt,
                                        int L, int Hq, int W, int32_t* __restrict__ vloc,
                                        int32_t* __restrict__ vcnt_loc) {
  __shared__ int wsum[32];
  __shared__ int carry_s;
  const int h = blockIdx.x % Hq, s = blockIdx.x / Hq;
  const int Ls = L / W;
  const int n = v_cnt[h];
  int32_t* out = vloc + ((size_t)s * Hq + h) * Ls;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  if (threadIdx.x == 0) carry_s = 0;
  __syncthreads();
  for (int base = 0; base < n; base += blockDim.x) {
    const int k = base + threadIdx.x;
    const int m = k < n ? v_idx[(size_t)h * L + k] : -1;
    const bool mine = m >= 0 && m < L && m % W == s;
    const unsigned b = __ballot_sync(0xffffffffu, mine);
    if (lane == 0) wsum[warp] = __popc(b);
    __syncthreads();
    int before = carry_s, total = 0;
    for (int q = 0; q < nw; ++q) {
      if (q < warp) before += wsum[q];
      total += wsum[q];
    }
    if (mine) out[before + __popc(b & ((1u << lane) - 1u))] = m / W;
    __syncthreads();
    if (threadIdx.x == 0) carry_s += total;
    __syncthreads();
  }
  if (threadIdx.x == 0) vcnt_loc[(size_t)s * Hq + h] = carry_s;
}

// fp32 sums -> bf16 (dK, dV of the ring backward)
__global__ void ring_finish_kernel(const float* __restrict__ a, __nv_bfloat16* __restrict__ out, long long n) {
  const long long i = ((long long)blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (i + 3 < n) {
    const float4 v = *reinterpret_cast<const float4*>(a + i);
    uint2 o;
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
    o.x = *reinterpret_cast<uint32_t*>(&lo);
    o.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(out + i) = o;
  } else {
    for (long long k = i; k < n; ++k) out[k] = __float2bfloat16_rn(a[k]);
  }
}

struct RingWs {
  size_t status, vloc, vcnt, inS, shard0, shard_stride, carry_o, carry_lse2;  // forward and backward
  size_t dsum, part_k, part_v, dk32, dv32;                                   // backward only
  size_t total;
  PrepWs shard;  // offsets of one shard's prep regions relative to its start
};

// local geometry of the steps
vs_params local_params(const vs_params& p) {
  vs_params q = p;
  q.L = p.L / p.stripes;
  q.stripes = 1;
  return q;
}

RingWs ring_layout(const vs_params& p, bool bwd) {
  const int W = p.stripes;
  const vs_params pl = local_params(p);
  const AttnGeom gl = make_geom(pl);
  RingWs o;
  WsLayout w;
  o.status = w.take(sizeof(DevStatus));
  o.vloc = w.take((size_t)W * p.Hq * gl.L * 4);
  o.vcnt = w.take((size_t)W * p.Hq * 4);
  o.inS = w.take((size_t)p.Hq * gl.nw * 4);
  // one shard's prep regions (the kept-band bitmaps are shared: inS above)
  WsLayout ws1;
  o.shard = prep_layout(gl, ws1);
  o.shard_stride = align_up(ws1.off, 256);
  o.shard0 = w.take(o.shard_stride * W);
  o.carry_o = w.take((size_t)gl.L * p.Hq * p.d * 4);
  o.carry_lse2 = bwd ? w.off : w.take((size_t)p.Hq * gl.L * 4);
  o.dsum = o.part_k = o.part_v = o.dk32 = o.dv32 = w.off;
  if (bwd) {
    o.dsum = w.take((size_t)p.Hq * p.L * 4);
    o.part_k = w.take(bwd_partials_bytes(gl));
    o.part_v = w.take(bwd_partials_bytes(gl));
    o.dk32 = w.take((size_t)p.L * p.Hkv * p.d * 4);
    o.dv32 = w.take((size_t)p.L * p.Hkv * p.d * 4);
  }
  o.total = w.off;
  return o;
}

struct RingCtx {
  vs_params pl;
  AttnGeom gl;
  uint8_t* w;
  RingWs lay;
  int W;
};

PrepPtrs shard_prep(const RingCtx& c, int s) {
  uint8_t* b = c.w + c.lay.shard0 + (size_t)s * c.lay.shard_stride;
  PrepPtrs pp;
  pp.inS = reinterpret_cast<uint32_t*>(c.w + c.lay.inS);
  pp.vlist = reinterpret_cast<uint32_t*>(b + c.lay.shard.vlist);
  pp.vcnt = reinterpret_cast<int32_t*>(b + c.lay.shard.vcnt);
  pp.Kp = reinterpret_cast<__nv_bfloat16*>(b + c.lay.shard.Kp);
  pp.Vp = reinterpret_cast<__nv_bfloat16*>(b + c.lay.shard.Vp);
  pp.vbits = c.lay.shard.vbits != c.lay.shard.end ? reinterpret_cast<uint32_t*>(b + c.lay.shard.vbits) : nullptr;
  return pp;
}

vs_index shard_index(const RingCtx& c, const vs_index& ix, int s) {
  vs_index o = ix;
  o.v_idx = reinterpret_cast<int32_t*>(c.w + c.lay.vloc) + (size_t)s * c.pl.Hq * c.gl.L;
  o.v_cnt = reinterpret_cast<int32_t*>(c.w + c.lay.vcnt) + (size_t)s * c.pl.Hq;
  o.v_score = o.s_score = nullptr;
  o.active_entries = nullptr;
  return o;
}

AttnGeom step_geom(const RingCtx& c, int r, int s) {
  AttnGeom g = c.gl;
  g.L_glob = c.gl.L * c.W;
  g.tq_mul = g.tk_mul = c.W;
  g.tq_add = r;
  g.tk_add = s;
  g.strict_diag = s > r ? 1 : 0;
  return g;
}

// shard vertical lists, shared band bitmaps, per-shard vertical unions and packed rows
cudaError_t ring_setup(const RingCtx& c, const vs_index& ix, const void* K, const void* V, cudaStream_t st) {
  const int Hq = c.pl.Hq, W = c.W;
  ring_shard_index_kernel<<<Hq * W, 256, 0, st>>>(ix.v_idx, ix.v_cnt, c.gl.L * W, Hq, W,
                                                  reinterpret_cast<int32_t*>(c.w + c.lay.vloc),
                                                  reinterpret_cast<int32_t*>(c.w + c.lay.vcnt));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if ((e = launch_prep_bands(c.gl, ix, shard_prep(c, 0), st)) != cudaSuccess) return e;
  for (int s = 0; s < W; ++s) {
    AttnGeom g = c.gl;
    g.L_glob = c.gl.L * W;
    g.tk_mul = W;
    g.tk_add = s;
    if ((e = launch_prep_verticals(g, shard_index(c, ix, s), K, V, shard_prep(c, s), st)) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

int step_mode(int t, int W) {
  if (W == 1) return kAccPlain;
  return t == 0 ? kAccFirst : (t == W - 1 ? kAccLast : kAccMid);
}

cudaError_t record(void* const* ev, int n_ev, int k, cudaStream_t st) {
  if (!ev || k >= n_ev) return cudaSuccess;
  return cudaEventRecord(static_cast<cudaEvent_t>(ev[k]), st);
}

}  // namespace

size_t ring_ws_bytes(const vs_params& p, bool bwd) { return ring_layout(p, bwd).total; }

cudaError_t launch_ring_fwd(const vs_params& p, const vs_index& ix, const void* Q, const void* K, const void* V,
                            void* O, float* lse, void* ws, void* const* ev, int n_ev, cudaStream_t st) {
  RingCtx c;
  c.pl = local_params(p);
  c.gl = make_geom(c.pl);
  c.w = static_cast<uint8_t*>(ws);
  c.lay = ring_layout(p, false);
  c.W = p.stripes;
  cudaError_t e = ring_setup(c, ix, K, V, st);
  if (e != cudaSuccess) return e;
  DevStatus* status = reinterpret_cast<DevStatus*>(c.w + c.lay.status);
  StepCtl ctl;
  ctl.carry_o = reinterpret_cast<float*>(c.w + c.lay.carry_o);
  ctl.carry_lse2 = reinterpret_cast<float*>(c.w + c.lay.carry_lse2);
  for (int r = 0; r < c.W; ++r)
    for (int t = 0; t < c.W; ++t) {
      const int s = (r - t + c.W) % c.W;
      if ((e = record(ev, n_ev, r * c.W + t, st)) != cudaSuccess) return e;
      ctl.acc_mode = step_mode(t, c.W);
      if ((e = launch_fwd_core(c.pl, step_geom(c, r, s), shard_prep(c, s), Q, K, V, O, lse, status, ctl, st)) !=
          cudaSuccess)
        return e;
    }
  return record(ev, n_ev, c.W * c.W, st);
}

cudaError_t launch_ring_bwd(const vs_params& p, const vs_index& ix, const void* Q, const void* K, const void* V,
                            const void* O, const float* lse, const void* dO, void* dQ, void* dK, void* dV, void* ws,
                            void* const* ev, int n_ev, cudaStream_t st) {
  if (p.d != 128) return cudaErrorNotSupported;
  RingCtx c;
  c.pl = local_params(p);
  c.gl = make_geom(c.pl);
  c.w = static_cast<uint8_t*>(ws);
  c.lay = ring_layout(p, true);
  c.W = p.stripes;
  cudaError_t e = ring_setup(c, ix, K, V, st);
  if (e != cudaSuccess) return e;
  DevStatus* status = reinterpret_cast<DevStatus*>(c.w + c.lay.status);
  float* dsum = reinterpret_cast<float*>(c.w + c.lay.dsum);
  float* dk32 = reinterpret_cast<float*>(c.w + c.lay.dk32);
  float* dv32 = reinterpret_cast<float*>(c.w + c.lay.dv32);
  const size_t nkv = (size_t)p.L * p.Hkv * p.d;
  if ((e = launch_bwd_dsum(O, dO, dsum, p.L, p.Hq, p.d, st)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(dk32, 0, nkv * 4, st)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(dv32, 0, nkv * 4, st)) != cudaSuccess) return e;
  StepCtl ctl;
  ctl.carry_o = reinterpret_cast<float*>(c.w + c.lay.carry_o);
  for (int r = 0; r < c.W; ++r)
    for (int t = 0; t < c.W; ++t) {
      const int s = (r - t + c.W) % c.W;
      if ((e = record(ev, n_ev, r * c.W + t, st)) != cudaSuccess) return e;
      const AttnGeom g = step_geom(c, r, s);
      const PrepPtrs pp = shard_prep(c, s);
      if ((e = launch_dkdv_core(c.pl, g, pp, shard_index(c, ix, s), Q, K, V, dO, lse, dsum, dK, dV,
                                reinterpret_cast<float*>(c.w + c.lay.part_k),
                                reinterpret_cast<float*>(c.w + c.lay.part_v), dk32, dv32, status, nullptr, st)) !=
          cudaSuccess)
        return e;
      ctl.acc_mode = step_mode(t, c.W);
      if ((e = launch_attn_dq(c.pl, g, pp, Q, K, V, dO, lse, dsum, dQ, status, ctl, st)) != cudaSuccess) return e;
    }
  if ((e = record(ev, n_ev, c.W * c.W, st)) != cudaSuccess) return e;
  const unsigned nb = (unsigned)((nkv / 4 + 255) / 256);
  ring_finish_kernel<<<nb, 256, 0, st>>>(dk32, static_cast<__nv_bfloat16*>(dK), (long long)nkv);
  ring_finish_kernel<<<nb, 256, 0, st>>>(dv32, static_cast<__nv_bfloat16*>(dV), (long long)nkv);
  return cudaGetLastError();
}

}  // namespace vs
