// Shared definitions of the VS sparse attention library (host + device).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/vs.h"

namespace vs {

constexpr int kBlock = 64;                       // slash tile edge (keys and queries)
constexpr uint64_t kWaitLimitNs = 2000000000ull; // bounded in-kernel waits: 2 s
constexpr int kMaxL = 1 << 20;                   // supported sequence length ceiling

// Per-site wait-cycle and phase counters of the attention kernels are built
// only with -DVS_WAIT_PROFILE=n (a pipeline-balance diagnostic: 1 all
// attention kernels, 2 the dK/dV kernel, 3 the query-major kernel, 4 the
// dK/dV kernel's MMA issue only, 5 the query-major kernel's MMA issue
// only); the
// default build leaves the wait_cycles array of the status block at zero.
#ifndef VS_WAIT_PROFILE
#define VS_WAIT_PROFILE 0
#endif
constexpr bool kWaitProfileKv = VS_WAIT_PROFILE == 1 || VS_WAIT_PROFILE == 2;
// 7: the stored-dS dQ kernel's waits (producer, MMA issue, epilogue) and total cycles
constexpr bool kWaitProfileDs = VS_WAIT_PROFILE == 7;
// 8: the selection kernel's phases (budget fill), per head summed
constexpr bool kProfileSel = VS_WAIT_PROFILE == 8;
// 4: only the dK/dV kernel's MMA-issue timers and total cycles (least intrusive)
constexpr bool kMmaProfileKv = kWaitProfileKv || VS_WAIT_PROFILE == 4;
constexpr bool kWaitProfileQm = VS_WAIT_PROFILE == 1 || VS_WAIT_PROFILE == 3;
// 5: only the query-major kernel's MMA-issue timers and total cycles
constexpr bool kMmaProfileQm = kWaitProfileQm || VS_WAIT_PROFILE == 5 || VS_WAIT_PROFILE == 6;
// 6: additionally the softmax warps' per-tile wait / work split, kept in registers
constexpr bool kSmProfileQm = VS_WAIT_PROFILE == 6;

// Device-side status block (first bytes of every workspace).
constexpr int kWaitSites = 32;
struct DevStatus {
  int32_t code;   // VS_OK or VS_ERR_TIMEOUT
  int32_t where;  // a wait that gave up: kernel tag * 100 + wait site
  int32_t path;   // backward: 1 when dQ was formed from stored dS tiles
  int32_t passes; // backward: the stored-dS passes that ran (key/value head groups split)
  // Cycles spent blocked at each wait site of the attention kernels, summed
  // over CTAs (lane 0 of each waiting warp), and the kernels' total cycles
  // per CTA in slot 31: a pipeline-balance diagnostic read by profiling tools.
  unsigned long long wait_cycles[kWaitSites];
};

// Bounded-wait test hook, read from the environment by the launchers (unset
// in normal use):
//   VS_TEST_STALL_PRODUCERS=1  the dK / dV kernel's planner, and the
//                              producers of a ring step's query-major kernel,
//                              are given no work: they issue no copy and
//                              arrive on no barrier, and every consumer's
//                              first wait runs out after the 2 s limit (no
//                              copy or MMA is ever in flight).
// The kernels then record VS_ERR_TIMEOUT, free their tensor memory and
// return; vs_device_status reports it.  The hook reaches the kernels as a
// parameter read once per warp (a loop bound in the query-major kernel's
// ring-step instance only, so a plain call's code carries nothing for it).
bool test_stall_requested();

// Device bounds checks of a VS_DEBUG build (-DVS_DEBUG=1): VS_BOUNDS(cond,
// st, site) is true when cond holds; otherwise it records VS_ERR_BOUNDS and
// the site in the status block (once; no trap) and is false, so the caller
// skips the access.  In a normal build it is the constant true and the check
// compiles away.
#ifndef VS_DEBUG
#define VS_DEBUG 0
#endif
__device__ __forceinline__ bool report_bounds(DevStatus* st, int site) {
  if (st && atomicCAS(&st->code, (int32_t)VS_OK, (int32_t)VS_ERR_BOUNDS) == (int32_t)VS_OK) atomicExch(&st->where, site);
  return false;
}
#if VS_DEBUG
#define VS_BOUNDS(cond, st, site) ((cond) ? true : ::vs::report_bounds((st), (site)))
#else
#define VS_BOUNDS(cond, st, site) true
#endif

// Records a wait that gave up: `where` = kernel tag * 100 + the kernel's
// wait site (when several give up, one of them).
__device__ __forceinline__ void report_timeout(DevStatus* st, int where) {
  if (st) {
    atomicExch(&st->code, (int32_t)VS_ERR_TIMEOUT);
    atomicExch(&st->where, where);
  }
}
// The same, keeping the first wait that gave up (the dK / dV kernel; the
// query-major kernel's register budget has no room for the compare).
__device__ __forceinline__ void report_timeout_first(DevStatus* st, int where) {
  if (st && atomicCAS(&st->code, (int32_t)VS_OK, (int32_t)VS_ERR_TIMEOUT) == (int32_t)VS_OK)
    atomicExch(&st->where, where);
}
// kernel tags of the status word's wait site
enum : int {
  kTagForward = 1, kTagDq = 2, kTagDkdvVertical = 3, kTagDkdvSlash = 4, kTagDqStored = 5, kTagIndex = 6,
  kTagXattn = 7
};

__host__ __device__ constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Simple bump allocator over the caller's workspace (host side, computes offsets only).
struct WsLayout {
  size_t off = 0;
  size_t take(size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  }
};

inline float default_scale(const vs_params& p) {
  return p.softmax_scale > 0.f ? p.softmax_scale : 1.0f / sqrtf((float)p.d);
}

// ---------------------------------------------------------------- launchers
// (implemented in the per-stage .cu files; all return cudaGetLastError())

struct RopeArgs {
  const void* x;
  void* y;
  int32_t L, H, d;
  int32_t transpose;
  float mscale;
  uint64_t turn[64];       // theta_i / (2 pi) as a 0.64 fixed-point fraction, d/2 <= 64 (host-computed in fp64)
  const int32_t* skip_if;  // device word or null: the kernel returns at once when it is non-zero
};
// The frequencies (rope_theta, YaRN) and temperature of p into a (x, y, L,
// H, transpose and skip_if are the caller's).
void rope_fill(const vs_params& p, RopeArgs& a);
cudaError_t launch_rope(const RopeArgs& a, cudaStream_t s);
// rope_mode = 1: the RoPE adjoint in place on dK [L][Hkv][d] and on dQ
// [L][Hq][d] (the dQ pass returns at once when *dq_skip_if != 0).
cudaError_t launch_rope_adjoint(const vs_params& p, void* dQ, void* dK, const int32_t* dq_skip_if, cudaStream_t s);

struct IndexArgs {
  const void* Q;
  const void* K;
  int32_t L, Hq, Hkv, G, d;
  int32_t last_q, qpad;       // index rows; rows per head padded to 16
  int32_t bs, nbs;            // slash tile (64 * stripes) and band count
  int32_t ntile;              // L / 64
  int32_t tiles_per_chunk, nchunk;
  int32_t row_splits;         // CTAs along the row dimension per KV head
  float scale_log2;           // softmax scale * log2(e)
  float top_p, density;
  float2* part;               // [nchunk][Hq*qpad] (max, sum) per chunk, log2 domain
  float2* rowstat;            // [Hq*qpad] (max, 1/sum)
  float* v;                   // [Hq][L]
  float* T64;                 // [Hq][last_q][ntile] row mass per 64-key tile
  float* S;                   // [Hq][nbs]
  int32_t* v_idx;
  int32_t* v_cnt;
  int32_t* s_idx;
  int32_t* s_cnt;
  int64_t* active;            // [Hq] or null
  uint32_t* vhist;            // [Hq][2048] counts of v by key >> 20 (written by the tensor-core
                              // pass 2), or null: the selection counts them itself
  DevStatus* status;
};
cudaError_t launch_index(const IndexArgs& a, cudaStream_t s);
// Key chunks and tiles of the tensor-core index passes (last_q = 64; the
// workspace sizes their partials array from it).
struct IxTcGrid {
  int C;       // key chunks
  int tpc;     // 128-key tiles per chunk
  int npairs;  // head pairs per key/value head
};
IxTcGrid index_tc_grid(int L, int Hq, int Hkv);
bool index_tc_supported(const IndexArgs& a);
void index_grid(const vs_params& p, int* tiles_per_chunk, int* nchunk, int* row_splits);

// Anti-diagonal block scorer (vs_xattn_index_build).
struct XaArgs {
  const void* Q;
  const void* K;
  int32_t L, Hq, Hkv, G, d;
  int32_t S, R, nrt;           // stride, strided rows L / S, 128-row tiles of them
  int32_t bs, bsS, nb, nw;     // block edge, strided rows per block, blocks per row, mask words per row
  float c2;                    // softmax scale * log2(e) / S
  float inv_bsS;
  float threshold;
  float2* rs;                  // [Hq][R] (max, sum) per strided row, log2 domain
  float* X;                    // [Hq][nb][nb] block scores
  uint32_t* mask;              // [Hq][nb][nw] kept-block bits
  int32_t* cnt;                // [Hq][nb] kept blocks per block row
  unsigned long long* active;  // [Hq] causal entries inside the kept blocks
  DevStatus* status;
};
cudaError_t launch_xattn(const XaArgs& a, cudaStream_t s);

}  // namespace vs
