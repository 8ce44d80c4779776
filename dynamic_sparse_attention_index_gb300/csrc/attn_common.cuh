// Work decomposition and preparation shared by the sparse attention forward
// and backward kernels.
//
// A row tile is 128 query rows = two 64-row "segments" (h_s, I_s) that use
// the same key/value head.  When the GQA group size G is even, a tile holds
// query block I of two heads of one group (their kept lines overlap heavily,
// so the union of their key sources wastes little); otherwise it holds
// blocks I and I+1 of one head.  A segment's active entries are
//   slash: key block kb with kb <= I_s and band I_s - kb kept for h_s
//          (band 0 = the diagonal block, causal inside);
//   vertical: kept token m of h_s with m/64 < I_s whose band I_s - m/64 is
//          not kept (otherwise the slash block already covers it).
// Key sources are 64-key units: one slash key block, or 64 consecutive
// entries of the tile's vertical union list (verticals of both segments'
// heads, ascending, with per-entry membership flags), whose K/V rows are
// packed contiguously by the prep kernels so TMA can stage them.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>

#include "common.cuh"

namespace vs {

constexpr uint32_t kVFlagShift = 30;  // union entry = token | (membership bits << 30)
constexpr uint32_t kVTokenMask = (1u << kVFlagShift) - 1u;

struct AttnGeom {
  int L, Hq, Hkv, G, d;
  int nb;           // L / 64 query / key blocks
  int nbs;          // L / bs (bands)
  int bs;           // 64 * stripes
  int nw;           // 32-bit words per kept-band bitmap (covers nbs bands)
  int pair_heads;   // 1: tiles pair two heads at the same block; 0: blocks I, I+1 of one head
  int nvg;          // vertical union groups (head pairs, or heads)
  int nitems;       // row tiles
  int items_per_row;  // tiles per block index (pair_heads) or per block pair
  // One step of the striped sparse ring (worker r, KV shard s) runs as a
  // problem of L = L_glob / W local tokens: local query row i is global token
  // i * tq_mul + tq_add, local key row j is j * tk_mul + tk_add.  A plain call
  // has the identity maps and L_glob = L.
  int L_glob;       // global tokens: row stride of lse / D, token range of outputs
  int tq_mul, tq_add, tk_mul, tk_add;
  int strict_diag;  // 1: the diagonal tile admits key j only for j < i (KV shard after the worker's)
  __host__ __device__ int tq(int i) const { return i * tq_mul + tq_add; }
  __host__ __device__ int tk(int j) const { return j * tk_mul + tk_add; }
};

inline AttnGeom make_geom(const vs_params& p) {
  AttnGeom g;
  g.L = p.L;
  g.Hq = p.Hq;
  g.Hkv = p.Hkv;
  g.G = p.Hq / p.Hkv;
  g.d = p.d;
  g.nb = p.L / kBlock;
  g.bs = kBlock * p.stripes;
  g.nbs = p.L / g.bs;
  g.nw = (g.nbs + 31) / 32;
  g.pair_heads = (g.G % 2 == 0) ? 1 : 0;
  if (g.pair_heads) {
    g.nvg = p.Hq / 2;
    g.items_per_row = p.Hq / 2;
    g.nitems = g.nb * g.items_per_row;
  } else {
    g.nvg = p.Hq;
    g.items_per_row = p.Hq;
    g.nitems = ((g.nb + 1) / 2) * g.items_per_row;
  }
  g.L_glob = p.L;
  g.tq_mul = g.tk_mul = 1;
  g.tq_add = g.tk_add = 0;
  g.strict_diag = 0;
  return g;
}

// Active keys of the causal diagonal tile for row rr (keys 0..rr, or
// 0..rr-1 when the step's KV shard comes after the worker's own).
__host__ __device__ inline uint64_t diag_bits(int rr, int strict) {
  if (strict) return (1ull << rr) - 1ull;
  return rr >= 63 ? ~0ull : ((2ull << rr) - 1ull);
}

// Where a call's results go: written directly (a plain call), or one step
// of a ring whose partial results are carried across steps in fp32 scratch.
enum : int { kAccPlain = 0, kAccFirst = 1, kAccMid = 2, kAccLast = 3 };

struct Item {
  int g;        // key/value head
  int h[2];     // query heads of the two segments
  int I[2];     // query blocks (64 rows each)
  bool valid[2];
  int vg;       // vertical union group
};

// Items are numbered heaviest-first: larger block index = more causal keys.
// decode_item_at takes the item's row position (0 = heaviest) and its place
// pr in the row (0 .. items_per_row - 1).
__host__ __device__ inline Item decode_item_at(const AttnGeom& g, int row, int pr) {
  Item it;
  if (g.pair_heads) {
    const int I = g.nb - 1 - row;
    const int kv = pr / (g.G / 2), hp = pr % (g.G / 2);
    it.g = kv;
    it.h[0] = kv * g.G + 2 * hp;
    it.h[1] = it.h[0] + 1;
    it.I[0] = it.I[1] = I;
    it.valid[0] = it.valid[1] = true;
    it.vg = pr;
  } else {
    const int npair = (g.nb + 1) / 2;
    const int u = npair - 1 - row;
    const int h = pr;
    it.g = h / g.G;
    it.h[0] = it.h[1] = h;
    it.I[0] = 2 * u;
    it.I[1] = 2 * u + 1;
    it.valid[0] = true;
    it.valid[1] = (2 * u + 1) < g.nb;
    it.vg = h;
  }
  return it;
}
__host__ __device__ inline Item decode_item(const AttnGeom& g, int id) {
  return decode_item_at(g, id / g.items_per_row, id % g.items_per_row);
}
// Items of the key/value heads [kv_lo, kv_lo + kv_n) alone, numbered the same
// way (id < rows x kv_n x items_per_row / Hkv).
__host__ __device__ inline int items_per_kv(const AttnGeom& g) { return g.items_per_row / g.Hkv; }
__host__ __device__ inline Item decode_item_kv(const AttnGeom& g, int id, int kv_lo, int kv_n) {
  const int n = kv_n * items_per_kv(g);
  return decode_item_at(g, id / n, kv_lo * items_per_kv(g) + id % n);
}

// Workspace regions written by the prep kernels (offsets from ws base).
struct PrepWs {
  size_t inS;     // [Hq][nw] uint32 kept-band bitmaps
  size_t vlist;   // [nvg][L] uint32 union entries
  size_t vcnt;    // [nvg][nb + 1] int32: entries with token < 64 * b
  size_t Kp;      // [nvg][L][d] bf16 packed key rows of the union
  size_t Vp;      // [nvg][L][d] bf16 packed value rows
  size_t vbits;   // [nvg][2][L/32] uint32 per-head vertical bitmaps (when they exceed shared memory)
  size_t end;
};
// The vertical-union pass keeps two L-bit bitmaps per head pair; up to this
// many bytes they live in shared memory, beyond it in the workspace.
constexpr size_t kVunionSmemMax = 160 * 1024;

inline PrepWs prep_layout(const AttnGeom& g, WsLayout& w) {
  PrepWs o;
  o.inS = w.take((size_t)g.Hq * g.nw * 4);
  o.vlist = w.take((size_t)g.nvg * g.L * 4);
  o.vcnt = w.take((size_t)g.nvg * (g.nb + 1) * 4);
  o.Kp = w.take((size_t)g.nvg * g.L * g.d * 2);
  o.Vp = w.take((size_t)g.nvg * g.L * g.d * 2);
  o.vbits = w.take((size_t)2 * (g.L / 32) * 4 > kVunionSmemMax ? (size_t)g.nvg * 2 * (g.L / 32) * 4 : 0);
  o.end = w.off;
  return o;
}

struct PrepPtrs {
  uint32_t* inS;
  uint32_t* vlist;
  int32_t* vcnt;
  __nv_bfloat16* Kp;
  __nv_bfloat16* Vp;
  uint32_t* vbits;  // null when the bitmaps fit in shared memory
};

cudaError_t launch_attn_prep(const AttnGeom& g, const vs_index& ix, const void* K, const void* V,
                             const PrepPtrs& pp, cudaStream_t s);
// the kept-band bitmaps only, and the vertical union + packed rows only
cudaError_t launch_prep_bands(const AttnGeom& g, const vs_index& ix, const PrepPtrs& pp, cudaStream_t s);
cudaError_t launch_prep_verticals(const AttnGeom& g, const vs_index& ix, const void* K, const void* V,
                                  const PrepPtrs& pp, cudaStream_t s);

// How one launch of the query-major kernel stores its results: directly
// (kAccPlain) or as one step of a ring whose state is carried in fp32
// scratch between steps; and which row tiles it processes.
struct StepCtl {
  int acc_mode = kAccPlain;
  float* carry_o = nullptr;     // [L][Hq][d] local rows
  float* carry_lse2 = nullptr;  // [Hq][L] (forward)
  int item_lo = 0, item_hi = -1;  // -1: every row tile
  // the launch does nothing when this device word is non-zero (the stored
  // dS tiles of the backward fit, so the dQ kernel that reads them runs)
  const int32_t* skip_if = nullptr;
};

cudaError_t launch_fwd_core(const vs_params& p, const AttnGeom& g, const PrepPtrs& pp, const void* Q, const void* K,
                            const void* V, void* O, float* lse, DevStatus* st, const StepCtl& ctl, cudaStream_t s);
cudaError_t launch_attn_dq(const vs_params& p, const AttnGeom& g, const PrepPtrs& pp, const void* Q, const void* K,
                           const void* V, const void* dO, const float* lse, const float* Dsum, void* dQ,
                           DevStatus* st, const StepCtl& ctl, cudaStream_t s);

// Stored dS tiles of the backward.  When the caller's workspace has room,
// the key-stationary dK / dV kernel writes every 64 x 64 dS block it forms
// (dS = P (dP - D), bf16, 64 query rows x 64 keys, keys contiguous) and the
// dQ kernel reads them back instead of recomputing S and dP.  The blocks of
// (query head h, query block I) follow that row's key sources in order: the
// slash key blocks active for h in descending key order (band 0, then each
// kept band B >= 1 ascending), then the 64-entry chunks of the vertical
// union list.  The backward runs in passes over whole key/value head groups
// (hpp = heads per pass, a multiple of Hq / Hkv; one pass when everything
// fits): the blocks of one pass's heads are stored and read back before the
// next pass reuses the room, and head h owns blocks [(h mod hpp) cap,
// (h mod hpp + 1) cap); one more block after them holds zeros.
struct DsPlan {
  int32_t* ok;         // device word: non-zero while every head's blocks fit in cap
  int32_t* band_rank;  // [Hq][nbs]: kept bands of head h in [1, B]
  int32_t* base_s;     // [Hq][nb]: first block of (h, I)
  int32_t* base_v;     // [Hq][nb]: first vertical-chunk block of (h, I)
  __nv_bfloat16* ds;   // [hpp cap + 1][64][64] blocks
  int cap;             // blocks per head
  int hpp;             // query heads per pass
  int zero_blk;        // hpp cap: a block of zeros (the rows of a segment a source does not reach)
};
constexpr int kDsBlockBytes = 64 * 64 * 2;

// Block of slash key block kb for query block I of a head, where kb lies in
// band B (rank: the head's kept bands in [1, B]) and base is the first block
// of (h, I): band 0 holds I, I-1, ..., (I / W) W, and every kept band B >= 1
// the W blocks (I / W - B) W + W - 1 down to (I / W - B) W.
__host__ __device__ inline int ds_slash_block(const AttnGeom& g, int base, int rank, int B, int I, int kb) {
  const int W = g.bs / kBlock;
  if (B == 0) return base + (I - kb);
  const int Iw = I / W;
  return base + (I - Iw * W + 1) + W * (rank - 1) + ((Iw - B) * W + W - 1 - kb);
}

cudaError_t launch_ds_plan(const AttnGeom& g, const PrepPtrs& pp, const DsPlan& d, cudaStream_t s);
// dQ of the row tiles of key/value heads [kv_lo, kv_lo + kv_n) (one pass)
cudaError_t launch_dq_stored(const vs_params& p, const AttnGeom& g, const PrepPtrs& pp, const void* K,
                             const DsPlan& d, void* dQ, DevStatus* st, int kv_lo, int kv_n, cudaStream_t s);

// Tensor-map helpers (host): 3-D view (d, heads, tokens) of a [L][H][d] bf16
// tensor with a (64, 1, 64) box, and a 2-D view (d, rows) with a (64, 64) box,
// both with 128-byte swizzle (the tcgen05 K-major / MN-major SW128 layouts).
// make_map_heads can view every tok_mul-th token starting at tok_add (one
// shard of the striped layout) as L consecutive rows.
bool make_map_heads(CUtensorMap* m, const void* base, int L, int H, int d, int tok_mul = 1, int tok_add = 0);
bool make_map_rows(CUtensorMap* m, const void* base, long long rows, int d);
// make_map_strided views [L][H][d] with token t = c * S + j as element
// (channel, j * H + h, c): row c of the box at middle coordinate j * H + h is
// head h's token c * S + j (R = L / S rows).
bool make_map_strided(CUtensorMap* m, const void* base, int R, int H, int d, int S);

}  // namespace vs
