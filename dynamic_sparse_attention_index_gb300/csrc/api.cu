// extern "C" entry points of the VS sparse attention library: argument
// validation (host, before any launch), workspace layout, and launches.
#include <cmath>
#include <cstdlib>
#include <cstring>

#include <nvtx3/nvToolsExt.h>

#include "common.cuh"

namespace vs {

cudaError_t launch_index_scores(const IndexArgs& a, cudaStream_t s);
cudaError_t launch_select(const IndexArgs& a, cudaStream_t s);
size_t select_smem_bytes(int nbs);
size_t group_union_smem_bytes(int L, int bs);
cudaError_t launch_group_union(const vs_params& p, const vs_index& ix, cudaStream_t s);
cudaError_t launch_attn_fwd(const vs_params& p, const vs_index& ix, const void* Q, const void* K, const void* V,
                            void* O, float* lse, void* ws, cudaStream_t s, int blk_lo, int blk_hi);
size_t attn_fwd_ws_bytes(const vs_params& p);
cudaError_t launch_attn_bwd(const vs_params& p, const vs_index& ix, const void* Q, const void* K, const void* V,
                            const void* O, const float* lse, const void* dO, void* dQ, void* dK, void* dV, void* ws,
                            size_t ws_bytes, cudaStream_t s);
size_t attn_bwd_ws_bytes(const vs_params& p);
size_t attn_bwd_ws_bytes_stored(const vs_params& p);
size_t ring_ws_bytes(const vs_params& p, bool bwd);
cudaError_t launch_ring_fwd(const vs_params& p, const vs_index& ix, const void* Q, const void* K, const void* V,
                            void* O, float* lse, void* ws, void* const* ev, int n_ev, cudaStream_t st);
cudaError_t launch_ring_bwd(const vs_params& p, const vs_index& ix, const void* Q, const void* K, const void* V,
                            const void* O, const float* lse, const void* dO, void* dQ, void* dK, void* dV, void* ws,
                            void* const* ev, int n_ev, cudaStream_t st);

bool test_stall_requested() {
  const char* v = std::getenv("VS_TEST_STALL_PRODUCERS");
  return v && std::atoi(v) == 1;
}

namespace {

// An NVTX range around every entry point (a profiler shows each call of the
// library by name; without a tool attached a push / pop costs nanoseconds).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

vs_status check_params(const vs_params* p) {
  if (!p) return VS_ERR_INVALID_ARG;
  if (p->L <= 0 || p->Hq <= 0 || p->Hkv <= 0 || p->d <= 0) return VS_ERR_INVALID_ARG;
  if (p->Hq % p->Hkv != 0) return VS_ERR_INVALID_ARG;
  if (p->block != kBlock) return VS_ERR_UNSUPPORTED;
  if (p->stripes < 1) return VS_ERR_INVALID_ARG;
  if (p->L % (kBlock * p->stripes) != 0) return VS_ERR_INVALID_ARG;
  if (p->L > kMaxL) return VS_ERR_UNSUPPORTED;
  if (p->d != 64 && p->d != 128) return VS_ERR_UNSUPPORTED;
  if (p->last_q < 1 || p->last_q > p->L) return VS_ERR_INVALID_ARG;
  if (!(p->top_p > 0.f && p->top_p <= 1.f)) return VS_ERR_INVALID_ARG;
  if (!(p->density >= 0.f && p->density <= 1.f)) return VS_ERR_INVALID_ARG;
  if (!(p->softmax_scale >= 0.f) || !std::isfinite(p->softmax_scale)) return VS_ERR_INVALID_ARG;
  if (p->index_mode != 0 && p->index_mode != 1) return VS_ERR_INVALID_ARG;
  if (p->rope_mode != 0 && p->rope_mode != 1) return VS_ERR_INVALID_ARG;
  if (p->rope_mode == 1 &&
      (!(p->rope_theta > 1.0) || !(p->yarn_factor >= 1.f) || (p->yarn_factor > 1.f && p->yarn_orig_len <= 0)))
    return VS_ERR_INVALID_ARG;
  return VS_OK;
}

vs_status check_index_params(const vs_params* p) {
  vs_status st = check_params(p);
  if (st != VS_OK) return st;
  if (p->last_q > 256) return VS_ERR_UNSUPPORTED;  // index rows per head kept within one CTA
  return VS_OK;
}

struct IndexWs {
  size_t status, part, rowstat, v, T64, S, vhist, total;
};

IndexWs index_ws(const vs_params& p) {
  int tpc, nchunk, rs;
  index_grid(p, &tpc, &nchunk, &rs);
  // the tensor-core passes' key chunks (last_q = 64; two partials per chunk)
  // share the partials array
  const int ctc = 2 * index_tc_grid(p.L, p.Hq, p.Hkv).C;
  if (ctc > nchunk) nchunk = ctc;
  const size_t qpad = (size_t)(p.last_q + 15) / 16 * 16;
  const size_t bs = (size_t)kBlock * p.stripes;
  const size_t nbs = (size_t)p.L / bs;
  const size_t ntile = (size_t)p.L / kBlock;
  WsLayout w;
  IndexWs o;
  o.status = w.take(sizeof(DevStatus));
  o.part = w.take((size_t)nchunk * p.Hq * qpad * sizeof(float2));
  o.rowstat = w.take((size_t)p.Hq * qpad * sizeof(float2));
  o.v = w.take((size_t)p.Hq * p.L * sizeof(float));
  o.T64 = w.take((size_t)p.Hq * p.last_q * ntile * sizeof(float));
  o.S = w.take((size_t)p.Hq * nbs * sizeof(float));
  o.vhist = w.take((size_t)p.Hq * 2048 * sizeof(uint32_t));
  o.total = w.off;
  return o;
}

struct XattnWs {
  size_t status, rs, cnt, active, total;
};

// Sized for any stride (stride 1 has the most strided rows, L per head).
XattnWs xattn_ws(const vs_params& p) {
  const size_t nb = (size_t)p.L / ((size_t)kBlock * p.stripes);
  WsLayout w;
  XattnWs o;
  o.status = w.take(sizeof(DevStatus));
  o.rs = w.take((size_t)p.Hq * p.L * sizeof(float2));
  o.cnt = w.take((size_t)p.Hq * nb * sizeof(int32_t));
  o.active = w.take((size_t)p.Hq * sizeof(unsigned long long));
  o.total = w.off;
  return o;
}

vs_status check_ws(const void* ws, size_t ws_bytes, size_t need) {
  if (!ws) return VS_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return VS_ERR_WORKSPACE;
  if (ws_bytes < need) return VS_ERR_WORKSPACE;
  return VS_OK;
}

vs_status check_index_ptrs(const vs_index* ix) {
  if (!ix || !ix->v_idx || !ix->v_cnt || !ix->s_idx || !ix->s_cnt) return VS_ERR_INVALID_ARG;
  // every data pointer 16-byte aligned (the selection reads v_score as 16-byte vectors)
  const void* ptrs[] = {ix->v_idx, ix->v_cnt, ix->s_idx, ix->s_cnt, ix->v_score, ix->s_score, ix->active_entries};
  for (const void* q : ptrs)
    if (q && !aligned16(q)) return VS_ERR_INVALID_ARG;
  return VS_OK;
}

}  // namespace
}  // namespace vs

using namespace vs;

extern "C" {

const char* vs_status_string(vs_status s) {
  switch (s) {
    case VS_OK: return "VS_OK";
    case VS_ERR_INVALID_ARG: return "VS_ERR_INVALID_ARG: invalid argument";
    case VS_ERR_UNSUPPORTED: return "VS_ERR_UNSUPPORTED: unsupported configuration";
    case VS_ERR_WORKSPACE: return "VS_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case VS_ERR_CUDA: return "VS_ERR_CUDA: CUDA launch or runtime error";
    case VS_ERR_TIMEOUT: return "VS_ERR_TIMEOUT: a bounded in-kernel wait gave up";
    case VS_ERR_BOUNDS: return "VS_ERR_BOUNDS: a device bounds check failed (VS_DEBUG build)";
  }
  return "VS_ERR_UNKNOWN";
}

size_t vs_workspace_bytes(const vs_params* p, int op) {
  if (op == VS_OP_ROPE) return 0;
  if (op == VS_OP_INDEX) {
    if (check_index_params(p) != VS_OK) return 0;
    return index_ws(*p).total;
  }
  if (check_params(p) != VS_OK) return 0;
  if (op == VS_OP_FWD) return attn_fwd_ws_bytes(*p);
  if (op == VS_OP_BWD) return p->d == 128 ? attn_bwd_ws_bytes_stored(*p) : 0;
  if (op == VS_OP_BWD_MIN) return p->d == 128 ? attn_bwd_ws_bytes(*p) : 0;
  if (op == VS_OP_RING_FWD) return ring_ws_bytes(*p, false);
  if (op == VS_OP_RING_BWD) return p->d == 128 ? ring_ws_bytes(*p, true) : 0;
  if (op == VS_OP_XATTN) return xattn_ws(*p).total;
  return 0;
}

vs_status vs_rope(const vs_params* p, int32_t H, const void* x, void* y, int32_t transpose, void* stream) {
  NvtxRange nvtx("vs_rope");
  if (!p || !x || !y || H <= 0 || p->L <= 0) return VS_ERR_INVALID_ARG;
  if (p->d != 64 && p->d != 128) return VS_ERR_UNSUPPORTED;
  if (!(p->rope_theta > 1.0) || !(p->yarn_factor >= 1.f)) return VS_ERR_INVALID_ARG;
  if (p->yarn_factor > 1.f && p->yarn_orig_len <= 0) return VS_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y)) return VS_ERR_INVALID_ARG;
  RopeArgs a;
  std::memset(&a, 0, sizeof(a));
  a.x = x;
  a.y = y;
  a.L = p->L;
  a.H = H;
  a.d = p->d;
  a.transpose = transpose ? 1 : 0;
  rope_fill(*p, a);
  return launch_rope(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? VS_OK : VS_ERR_CUDA;
}

vs_status vs_index_build(const vs_params* p, const void* Q, const void* K, const vs_index* out, void* ws,
                         size_t ws_bytes, void* stream) {
  NvtxRange nvtx("vs_index_build");
  vs_status st = check_index_params(p);
  if (st != VS_OK) return st;
  if (!Q || !K || !aligned16(Q) || !aligned16(K)) return VS_ERR_INVALID_ARG;
  if ((st = check_index_ptrs(out)) != VS_OK) return st;
  const IndexWs lay = index_ws(*p);
  if ((st = check_ws(ws, ws_bytes, lay.total)) != VS_OK) return st;
  // every host-side check comes before the first enqueue: a rejected call
  // leaves the stream and the workspace untouched
  const int nbs_check = p->L / (kBlock * p->stripes);
  if (select_smem_bytes(nbs_check) + 26 * 1024 > 227 * 1024) return VS_ERR_UNSUPPORTED;
  if (p->index_mode == 1 && group_union_smem_bytes(p->L, kBlock * p->stripes) > 227 * 1024 - 2048)
    return VS_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  if (cudaMemsetAsync(w + lay.status, 0, sizeof(DevStatus), s) != cudaSuccess) return VS_ERR_CUDA;

  IndexArgs a;
  std::memset(&a, 0, sizeof(a));
  a.Q = Q;
  a.K = K;
  a.L = p->L;
  a.Hq = p->Hq;
  a.Hkv = p->Hkv;
  a.G = p->Hq / p->Hkv;
  a.d = p->d;
  a.last_q = p->last_q;
  a.qpad = (p->last_q + 15) / 16 * 16;
  a.bs = kBlock * p->stripes;
  a.nbs = p->L / a.bs;
  a.ntile = p->L / kBlock;
  index_grid(*p, &a.tiles_per_chunk, &a.nchunk, &a.row_splits);
  a.scale_log2 = default_scale(*p) * 1.4426950408889634f;
  a.top_p = p->top_p;
  a.density = p->density;
  a.part = reinterpret_cast<float2*>(w + lay.part);
  a.rowstat = reinterpret_cast<float2*>(w + lay.rowstat);
  a.v = out->v_score ? out->v_score : reinterpret_cast<float*>(w + lay.v);
  a.T64 = reinterpret_cast<float*>(w + lay.T64);
  a.S = out->s_score ? out->s_score : reinterpret_cast<float*>(w + lay.S);
  a.v_idx = out->v_idx;
  a.v_cnt = out->v_cnt;
  a.s_idx = out->s_idx;
  a.s_cnt = out->s_cnt;
  a.active = out->active_entries;
  a.status = reinterpret_cast<DevStatus*>(w + lay.status);
  // cleared and filled by the tensor-core scoring passes; the others leave
  // the counting to the selection
  a.vhist = index_tc_supported(a) ? reinterpret_cast<uint32_t*>(w + lay.vhist) : nullptr;
  if (launch_index_scores(a, s) != cudaSuccess) return VS_ERR_CUDA;
  if (launch_select(a, s) != cudaSuccess) return VS_ERR_CUDA;
  if (p->index_mode == 1 && launch_group_union(*p, *out, s) != cudaSuccess) return VS_ERR_CUDA;
  return VS_OK;
}

vs_status vs_xattn_index_build(const vs_params* p, int32_t stride, float threshold, const void* Q, const void* K,
                               const vs_xattn_index* out, void* ws, size_t ws_bytes, void* stream) {
  NvtxRange nvtx("vs_xattn_index_build");
  vs_status st = check_params(p);
  if (st != VS_OK) return st;
  if (!Q || !K || !aligned16(Q) || !aligned16(K)) return VS_ERR_INVALID_ARG;
  if (!out || !out->block_score || !out->block_mask) return VS_ERR_INVALID_ARG;
  const void* ptrs[] = {out->block_score, out->block_mask, out->block_cnt, out->active_entries};
  for (const void* q : ptrs)
    if (q && !aligned16(q)) return VS_ERR_INVALID_ARG;
  if (!(threshold > 0.f && threshold <= 1.f)) return VS_ERR_INVALID_ARG;
  const int bs = kBlock * p->stripes;
  // the stride divides the block edge; a block has 4 .. 128 strided rows
  if (stride < 1 || (stride & (stride - 1)) != 0 || bs % stride != 0) return VS_ERR_INVALID_ARG;
  const int bsS = bs / stride;
  if (bsS < 4 || bsS > 128 || (bsS & (bsS - 1)) != 0) return VS_ERR_UNSUPPORTED;
  const int nb = p->L / bs;
  const XattnWs lay = xattn_ws(*p);
  if ((st = check_ws(ws, ws_bytes, lay.total)) != VS_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  if (cudaMemsetAsync(w + lay.status, 0, sizeof(DevStatus), s) != cudaSuccess) return VS_ERR_CUDA;
  XaArgs a;
  std::memset(&a, 0, sizeof(a));
  a.Q = Q;
  a.K = K;
  a.L = p->L;
  a.Hq = p->Hq;
  a.Hkv = p->Hkv;
  a.G = p->Hq / p->Hkv;
  a.d = p->d;
  a.S = stride;
  a.R = p->L / stride;
  a.nrt = (a.R + 127) / 128;
  a.bs = bs;
  a.bsS = bsS;
  a.nb = nb;
  a.nw = (nb + 31) / 32;
  a.c2 = default_scale(*p) * 1.4426950408889634f / (float)stride;
  a.inv_bsS = 1.0f / (float)bsS;
  a.threshold = threshold;
  a.rs = reinterpret_cast<float2*>(w + lay.rs);
  a.X = out->block_score;
  a.mask = out->block_mask;
  a.cnt = out->block_cnt ? out->block_cnt : reinterpret_cast<int32_t*>(w + lay.cnt);
  a.active = out->active_entries ? reinterpret_cast<unsigned long long*>(out->active_entries)
                                 : reinterpret_cast<unsigned long long*>(w + lay.active);
  a.status = reinterpret_cast<DevStatus*>(w + lay.status);
  return launch_xattn(a, s) == cudaSuccess ? VS_OK : VS_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// vs_index_build_noalloc: vs_index_build with library-owned scratch.
//
// Every other entry point takes its scratch from the caller.  This one is for
// callers that cannot provide it: code running where a device allocation is
// not allowed or not affordable at call time, e.g. a service whose caching
// allocator is already at its memory cap, a host program whose device
// footprint is planned once when the library loads, or a pipeline that must
// not stall (cudaMalloc and cudaFree synchronise the whole device).  Its
// scratch is a fixed-size array in the library's own device image, so no call
// allocates or frees anything.
}  // extern "C"

namespace {

// Holds the same layout as vs_index_build's caller workspace; problems whose
// workspace is larger are rejected.  Only the status block at its head must
// start at zero, and each call clears it on its stream first (inside
// vs_index_build); every other byte is written before it is read, so what an
// earlier call left behind does not matter.
static __device__ __align__(256) unsigned char g_index_scratch[VS_INDEX_NOALLOC_SCRATCH_BYTES];

// Host code sees g_index_scratch only as a host-side shadow symbol, never as
// a device address.  Every call resolves the array's address on the current
// device with cudaGetSymbolAddress (a host-side query that allocates
// nothing).  Nothing is cached, so the address stays right after a
// cudaDeviceReset or a change of the current device between calls.
vs_status noalloc_scratch(void** out) {
  void* a = nullptr;
  if (cudaGetSymbolAddress(&a, g_index_scratch) != cudaSuccess || !a) return VS_ERR_CUDA;
  *out = a;
  return VS_OK;
}

}  // namespace

extern "C" {

vs_status vs_index_build_noalloc(const vs_params* p, const void* Q, const void* K, const vs_index* out,
                                 void* stream) {
  NvtxRange nvtx("vs_index_build_noalloc");
  vs_status st = check_index_params(p);
  if (st != VS_OK) return st;
  if (!Q || !K || !aligned16(Q) || !aligned16(K)) return VS_ERR_INVALID_ARG;
  if ((st = check_index_ptrs(out)) != VS_OK) return st;
  if (index_ws(*p).total > (size_t)VS_INDEX_NOALLOC_SCRATCH_BYTES) return VS_ERR_WORKSPACE;
  void* scratch = nullptr;
  if ((st = noalloc_scratch(&scratch)) != VS_OK) return st;
  return vs_index_build(p, Q, K, out, scratch, (size_t)VS_INDEX_NOALLOC_SCRATCH_BYTES, stream);
}

vs_status vs_sparse_attn_fwd(const vs_params* p, const vs_index* index, const void* Q, const void* K,
                             const void* V, void* O, float* lse, void* ws, size_t ws_bytes, void* stream) {
  NvtxRange nvtx("vs_sparse_attn_fwd");
  vs_status st = check_params(p);
  if (st != VS_OK) return st;
  if ((st = check_index_ptrs(index)) != VS_OK) return st;
  if (!Q || !K || !V || !O || !lse) return VS_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(lse)) return VS_ERR_INVALID_ARG;
  if ((st = check_ws(ws, ws_bytes, attn_fwd_ws_bytes(*p))) != VS_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, sizeof(DevStatus), s) != cudaSuccess) return VS_ERR_CUDA;
  return launch_attn_fwd(*p, *index, Q, K, V, O, lse, ws, s, 0, p->L / kBlock) == cudaSuccess ? VS_OK : VS_ERR_CUDA;
}

vs_status vs_sparse_attn_fwd_rows(const vs_params* p, const vs_index* index, const void* Q, const void* K,
                                  const void* V, void* O, float* lse, void* ws, size_t ws_bytes, int32_t row_lo,
                                  int32_t row_hi, void* stream) {
  NvtxRange nvtx("vs_sparse_attn_fwd_rows");
  vs_status st = check_params(p);
  if (st != VS_OK) return st;
  if (row_lo < 0 || row_hi > p->L || row_lo >= row_hi || row_lo % kBlock || row_hi % kBlock)
    return VS_ERR_INVALID_ARG;
  if ((st = check_index_ptrs(index)) != VS_OK) return st;
  if (!Q || !K || !V || !O || !lse) return VS_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(lse)) return VS_ERR_INVALID_ARG;
  if ((st = check_ws(ws, ws_bytes, attn_fwd_ws_bytes(*p))) != VS_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, sizeof(DevStatus), s) != cudaSuccess) return VS_ERR_CUDA;
  return launch_attn_fwd(*p, *index, Q, K, V, O, lse, ws, s, row_lo / kBlock, row_hi / kBlock) == cudaSuccess
             ? VS_OK
             : VS_ERR_CUDA;
}

vs_status vs_sparse_attn_bwd(const vs_params* p, const vs_index* index, const void* Q, const void* K,
                             const void* V, const void* O, const float* lse, const void* dO, void* dQ,
                             void* dK, void* dV, void* ws, size_t ws_bytes, void* stream) {
  NvtxRange nvtx("vs_sparse_attn_bwd");
  vs_status st = check_params(p);
  if (st != VS_OK) return st;
  if ((st = check_index_ptrs(index)) != VS_OK) return st;
  if (p->d != 128) return VS_ERR_UNSUPPORTED;  // the backward kernels are built for d = 128
  if (!Q || !K || !V || !O || !lse || !dO || !dQ || !dK || !dV) return VS_ERR_INVALID_ARG;
  const void* ptrs[] = {Q, K, V, O, lse, dO, dQ, dK, dV};
  for (const void* q : ptrs)
    if (!aligned16(q)) return VS_ERR_INVALID_ARG;
  if ((st = check_ws(ws, ws_bytes, attn_bwd_ws_bytes(*p))) != VS_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, sizeof(DevStatus), s) != cudaSuccess) return VS_ERR_CUDA;
  return launch_attn_bwd(*p, *index, Q, K, V, O, lse, dO, dQ, dK, dV, ws, ws_bytes, s) == cudaSuccess ? VS_OK
                                                                                         : VS_ERR_CUDA;
}

vs_status vs_striped_ring_fwd(const vs_params* p, const vs_index* index, const void* Q, const void* K,
                              const void* V, void* O, float* lse, void* ws, size_t ws_bytes, void* const* step_events,
                              int32_t n_events, void* stream) {
  NvtxRange nvtx("vs_striped_ring_fwd");
  vs_status st = check_params(p);
  if (st != VS_OK) return st;
  if ((st = check_index_ptrs(index)) != VS_OK) return st;
  if (!Q || !K || !V || !O || !lse) return VS_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(lse)) return VS_ERR_INVALID_ARG;
  if (n_events < 0 || (n_events > 0 && !step_events)) return VS_ERR_INVALID_ARG;
  if ((st = check_ws(ws, ws_bytes, ring_ws_bytes(*p, false))) != VS_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, sizeof(DevStatus), s) != cudaSuccess) return VS_ERR_CUDA;
  return launch_ring_fwd(*p, *index, Q, K, V, O, lse, ws, step_events, n_events, s) == cudaSuccess ? VS_OK
                                                                                                  : VS_ERR_CUDA;
}

vs_status vs_striped_ring_bwd(const vs_params* p, const vs_index* index, const void* Q, const void* K,
                              const void* V, const void* O, const float* lse, const void* dO, void* dQ, void* dK,
                              void* dV, void* ws, size_t ws_bytes, void* const* step_events, int32_t n_events,
                              void* stream) {
  NvtxRange nvtx("vs_striped_ring_bwd");
  vs_status st = check_params(p);
  if (st != VS_OK) return st;
  if ((st = check_index_ptrs(index)) != VS_OK) return st;
  if (p->d != 128) return VS_ERR_UNSUPPORTED;
  if (!Q || !K || !V || !O || !lse || !dO || !dQ || !dK || !dV) return VS_ERR_INVALID_ARG;
  const void* ptrs[] = {Q, K, V, O, lse, dO, dQ, dK, dV};
  for (const void* q : ptrs)
    if (!aligned16(q)) return VS_ERR_INVALID_ARG;
  if (n_events < 0 || (n_events > 0 && !step_events)) return VS_ERR_INVALID_ARG;
  if ((st = check_ws(ws, ws_bytes, ring_ws_bytes(*p, true))) != VS_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, sizeof(DevStatus), s) != cudaSuccess) return VS_ERR_CUDA;
  if (launch_ring_bwd(*p, *index, Q, K, V, O, lse, dO, dQ, dK, dV, ws, step_events, n_events, s) != cudaSuccess)
    return VS_ERR_CUDA;
  // rope_mode = 1: the ring's dQ and dK back through the RoPE adjoint
  if (p->rope_mode == 1 && launch_rope_adjoint(*p, dQ, dK, nullptr, s) != cudaSuccess) return VS_ERR_CUDA;
  return VS_OK;
}

vs_status vs_device_status(void* ws, void* stream) {
  NvtxRange nvtx("vs_device_status");
  if (!ws) return VS_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return VS_ERR_CUDA;
  DevStatus h;
  if (cudaMemcpy(&h, ws, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return VS_ERR_CUDA;
  if (h.code == VS_OK) return VS_OK;
  if (cudaMemset(ws, 0, sizeof(DevStatus)) != cudaSuccess) return VS_ERR_CUDA;
  return (h.code == VS_ERR_TIMEOUT || h.code == VS_ERR_BOUNDS) ? (vs_status)h.code : VS_ERR_CUDA;
}

}  // extern "C"
