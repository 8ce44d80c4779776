/*
 * vs.h - C ABI of the GB300 (sm_103a) vertical-slash (VS) sparse attention library.
 *
 * The method (MTraining, arXiv 2510.18830; described in the paper review
 * "MTraining: 分布式动态稀疏注意力高效超长上下文训练", section 三 "技术架构"):
 *   1. online sparse-index approximation: the last `last_q` query rows are
 *      scored against every key, the softmax mass is summed along vertical
 *      lines (key token m) and slash bands (64x64 block diagonals), and the
 *      smallest sets of verticals and slashes that recall `top_p` of the mass
 *      are kept (section "分布式稀疏索引近似");
 *   2. block-sparse causal attention, forward and backward, over only the
 *      active entries, with an online softmax across key blocks (ring
 *      attention page, section 2.1 "块级循环计算范式").
 *
 * Conventions shared by every entry point
 *   - Tensors are token-major, batch 1: Q, O, dO, dQ are [L][Hq][d] and
 *     K, V, dK, dV are [L][Hkv][d], all bf16, rows packed (stride Hq*d or
 *     Hkv*d elements).  Every data pointer is a DEVICE pointer, 16-byte aligned.
 *   - The caller owns all memory.  The library never allocates or frees; the
 *     scratch an entry point needs is the caller's `ws` buffer of at least
 *     vs_workspace_bytes(...) bytes (256-byte aligned).
 *   - Every call is asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL = legacy default stream) and never synchronises.
 *   - Argument errors are detected on the host before any launch and returned
 *     as VS_ERR_INVALID_ARG / VS_ERR_UNSUPPORTED / VS_ERR_WORKSPACE; a failed
 *     launch returns VS_ERR_CUDA.  Kernels that wait on an in-CTA barrier do
 *     so for a bounded time; on timeout they record VS_ERR_TIMEOUT in the
 *     workspace status word (first 16 bytes of `ws`) and return, which
 *     vs_device_status() reports after the stream is synchronised.  After
 *     vs_sparse_attn_bwd, the status word's third int32 (bytes 8-11) is 1
 *     when dQ was formed from stored dS tiles and 0 when it was recomputed.
 *   - No global state, except the static scratch of vs_index_build_noalloc
 *     (see there): other calls on different streams with different
 *     workspaces are independent.
 */
#ifndef VS_H_
#define VS_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define VS_API __attribute__((visibility("default")))
#else
#define VS_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum vs_status {
  VS_OK = 0,
  VS_ERR_INVALID_ARG = 1, /* null pointer, out-of-range size or parameter */
  VS_ERR_UNSUPPORTED = 2, /* valid but not implemented (e.g. d not in {64,128}) */
  VS_ERR_WORKSPACE = 3,   /* ws too small or misaligned */
  VS_ERR_CUDA = 4,        /* a CUDA launch or runtime call failed */
  VS_ERR_TIMEOUT = 5,     /* a bounded in-kernel wait gave up (device-side) */
  VS_ERR_BOUNDS = 6       /* a device bounds check failed (VS_DEBUG builds only; device-side) */
} vs_status;

/* Problem description.  Batch 1. */
typedef struct vs_params {
  int32_t L;             /* tokens; multiple of 64 * stripes                         */
  int32_t Hq;            /* query heads                                              */
  int32_t Hkv;           /* key/value heads; Hq % Hkv == 0 (GQA group G = Hq/Hkv)     */
  int32_t d;             /* head dim: 64 or 128                                      */
  int32_t last_q;        /* index rows: the last last_q queries, 1 <= last_q <= L    */
  float top_p;           /* recall target per direction, 0 < top_p <= 1             */
  int32_t block;         /* slash tile edge; must be 64                              */
  int32_t stripes;       /* W >= 1: striped layout emulation (1 = contiguous)        */
  float softmax_scale;   /* 0 -> 1/sqrt(d)                                           */
  float density;         /* 0 -> top-p selection; in (0,1] -> budget fill to this    */
                         /*      active density (fixed-sparsity operating point)     */
  double rope_theta;     /* RoPE base (vs_rope only)                                 */
  float yarn_factor;     /* YaRN scale s (1 = plain RoPE)       (vs_rope only)       */
  int32_t yarn_orig_len; /* YaRN original context length        (vs_rope only)       */
  int32_t index_mode;    /* 0: one index per query head (the method);                */
                         /* 1: shared by each GQA group: every head of a key/value   */
                         /*    group uses the union of the group's per-head sets     */
                         /*    (vs_index_build; the attention calls read the arrays) */
  int32_t rope_mode;     /* 0: the backward's dQ, dK are gradients of the Q, K it    */
                         /*    was given (the rotated ones);                         */
                         /* 1: it maps them back through the RoPE adjoint of         */
                         /*    rope_theta / YaRN above: gradients of the un-rotated  */
                         /*    queries and keys (vs_sparse_attn_bwd and              */
                         /*    vs_striped_ring_bwd; Q and K are always passed        */
                         /*    rotated)                                               */
} vs_params;

/*
 * The sparse index, per query head h (all DEVICE pointers, caller-owned).
 * Slash band B of entry (n, m) is n/bs - m/bs with bs = block * stripes;
 * entry (n, m) is active iff m <= n and (band kept or m a kept vertical).
 */
typedef struct vs_index {
  int32_t* v_idx;          /* [Hq][L]     row h: v_cnt[h] ascending kept vertical token ids  */
  int32_t* v_cnt;          /* [Hq]                                                           */
  int32_t* s_idx;          /* [Hq][L/bs]  row h: s_cnt[h] ascending kept bands; band 0 kept  */
  int32_t* s_cnt;          /* [Hq]                                                           */
  float* v_score;          /* optional [Hq][L]    vertical mass (sum over the last_q rows)   */
  float* s_score;          /* optional [Hq][L/bs] slash-band mass                            */
  int64_t* active_entries; /* optional [Hq] exact active (n, m) entries per head             */
} vs_index;

/*
 * Block index of the anti-diagonal scorer (vs_xattn_index_build), per query
 * head h, with bs = block * stripes, nb = L / bs blocks per row and
 * nw = (nb + 31) / 32 mask words per block row (all DEVICE pointers,
 * caller-owned, 16-byte aligned).
 */
typedef struct vs_xattn_index {
  float* block_score;      /* [Hq][nb][nb] X[h][I][J]; zero above the diagonal (J > I)               */
  uint32_t* block_mask;    /* [Hq][nb][nw] bit J & 31 of word J >> 5 of row I: block (I, J) kept     */
  int32_t* block_cnt;      /* optional [Hq][nb] kept blocks of each block row (diagonal included)    */
  int64_t* active_entries; /* optional [Hq] causal (n, m) entries inside the kept blocks              */
} vs_xattn_index;

enum {
  VS_OP_INDEX = 0,
  VS_OP_FWD = 1,
  VS_OP_BWD = 2,     /* the backward with room for its stored dS tiles (see vs_sparse_attn_bwd) */
  VS_OP_ROPE = 3,
  VS_OP_RING_FWD = 4,
  VS_OP_RING_BWD = 5,
  VS_OP_BWD_MIN = 6, /* the least workspace vs_sparse_attn_bwd accepts (dS recomputed for dQ)   */
  VS_OP_XATTN = 7    /* vs_xattn_index_build (any stride)                                       */
};

/* Bytes of scratch `op` needs for problem `p` (0 if p is invalid). */
VS_API size_t vs_workspace_bytes(const vs_params* p, int op);

/* Human-readable name of a status code (static string). */
VS_API const char* vs_status_string(vs_status s);

/*
 * Rotate-half RoPE ("Vertical-Slash 稀疏模式" section: channel i pairs with
 * i + d/2, theta_i = rope_theta^(-2i/d); YaRN NTK-by-parts frequencies and
 * temperature when yarn_factor > 1).  x, y: [L][H][d] bf16, y may equal x.
 * transpose != 0 applies the adjoint (rotation by -phi), which maps the
 * gradient of a rotated tensor back to the un-rotated one.
 */
VS_API vs_status vs_rope(const vs_params* p, int32_t H, const void* x, void* y, int32_t transpose, void* stream);

/*
 * Sparse-index approximation ("分布式稀疏索引近似" section): scores the last
 * last_q rows of Q against all of K (scale * q.k, causal, softmax per row),
 * sums the probabilities per key (vertical) and per slash band, and keeps per
 * head the smallest descending prefix (ties: lower index) reaching top_p of
 * each direction's mass; band 0 is always kept.  With density > 0 the kept
 * set is instead the largest-mass candidates (verticals and bands ranked
 * together) whose active entries reach `density` of the causal entries.
 * With index_mode = 1 each head's lists and active count are then replaced
 * by those of the union over its GQA group (kernel-aware granularity
 * trade-off of the same section: fewer distinct index lines per key, more
 * entries); v_score / s_score stay per head.
 * Fills every non-NULL field of *out.
 */
VS_API vs_status vs_index_build(const vs_params* p, const void* Q, const void* K, const vs_index* out, void* ws,
                         size_t ws_bytes, void* stream);

/*
 * Anti-diagonal block index, an alternative to the vertical-slash index (the
 * ablation row "MTraining w/ XAttn Idx." of the MTraining review, section
 * 五 "实验结果", table "训练效率结果"; the pages only name it: this is the
 * published XAttention block scorer).  With S = stride, strided row r groups
 * query tokens rS .. rS+S-1 and strided column c key tokens cS .. cS+S-1;
 *   z[r, c] = scale / S * sum_j q[rS + j] . k[cS + S-1-j]   (the mean logit on
 *             the anti-diagonal of the S x S sub-block), cells c > r masked,
 *   P = softmax of z over each strided row,
 *   X[h][I][J] = (S / bs) * sum of P over the cells of block (I, J)
 *             (bs-token blocks; every block row sums to 1),
 * and each block row I keeps the smallest descending prefix of
 * X[h][I][0..I] (ties: lower J first) reaching `threshold` of the row's
 * total, plus the diagonal block I (threshold = 1 keeps every block of
 * positive score).  Uses L, Hq, Hkv, d, stripes (bs = 64 * stripes, the tile
 * of the striped-layout emulation) and softmax_scale of *p; Q [L][Hq][d] and
 * K [L][Hkv][d] bf16 as elsewhere.
 * Errors: VS_ERR_INVALID_ARG for a stride that is not a power of two
 * dividing bs, a threshold outside (0, 1] or a missing output;
 * VS_ERR_UNSUPPORTED unless 4 <= bs / stride <= 128.  Workspace:
 * vs_workspace_bytes(p, VS_OP_XATTN) bytes (any stride).  Fills every
 * non-NULL field of *out.
 */
VS_API vs_status vs_xattn_index_build(const vs_params* p, int32_t stride, float threshold, const void* Q,
                                      const void* K, const vs_xattn_index* out, void* ws, size_t ws_bytes,
                                      void* stream);

/*
 * Variant of vs_index_build that allocates nothing and takes no workspace.
 * The paper has no counterpart: this call exists for callers that cannot
 * give the library scratch memory at call time (e.g. code under an allocator
 * that is at its cap, code whose device footprint is fixed when the library
 * loads, or a pipeline that must not stall on cudaMalloc / cudaFree, which
 * synchronise the device).  Its scratch is one static device array of
 * VS_INDEX_NOALLOC_SCRATCH_BYTES (8 MiB) inside the library image, held by
 * every GPU that loads the library until the process exits; the call never
 * allocates or frees device memory.
 *   - Size limit: problems with vs_workspace_bytes(p, VS_OP_INDEX) above
 *     VS_INDEX_NOALLOC_SCRATCH_BYTES are rejected with VS_ERR_WORKSPACE
 *     before anything is launched (e.g. L = 32768, Hq = 16, last_q = 64
 *     needs 5 MiB and fits; L = 131072 with 16 heads does not).
 *   - Set-up: every call looks up the array's address on the current
 *     device (cudaGetSymbolAddress, a host-side query; nothing is cached,
 *     so a cudaDeviceReset between calls is harmless).  The first call on a
 *     device also loads the library's device code there: make that first
 *     call before any stream capture begins.
 *   - Zeroing: the array keeps what the last call left in it.  Only the
 *     status block at its head must start at zero, and every call clears it
 *     on `stream` before its kernels run.
 *   - Concurrency: all calls on one device share the one array.  Calls whose
 *     executions overlap on the GPU (different streams without an ordering
 *     between them, e.g. from several host threads) race on it and corrupt
 *     each other's results: issue them on one stream or order them with
 *     events.
 * Results, other arguments and other errors are exactly those of
 * vs_index_build.
 */
#define VS_INDEX_NOALLOC_SCRATCH_BYTES (8u << 20)
VS_API vs_status vs_index_build_noalloc(const vs_params* p, const void* Q, const void* K, const vs_index* out,
                                        void* stream);

/*
 * Block-sparse causal attention forward over the active entries of `index`
 * ("Ring Attention with sparse index" in the same section; online softmax
 * across key blocks): O = softmax(scale Q K^T restricted to the mask) V,
 * lse[h][n] = log sum_{m active} exp(scale q_n . k_m).
 * O: [L][Hq][d] bf16; lse: [Hq][L] fp32.
 */
VS_API vs_status vs_sparse_attn_fwd(const vs_params* p, const vs_index* index, const void* Q, const void* K,
                             const void* V, void* O, float* lse, void* ws, size_t ws_bytes, void* stream);

/*
 * vs_sparse_attn_fwd restricted to the query rows [row_lo, row_hi) (both
 * multiples of 64; the rows of every head): the same results for those rows,
 * the other rows of O and lse untouched.  A worker of a context-parallel
 * split that holds a range of query rows computes exactly this.  When
 * Hq / Hkv is odd, rows are processed in pairs of 64-row blocks, so the
 * range is widened to whole 128-row pairs.  Arguments and errors as
 * vs_sparse_attn_fwd; VS_ERR_INVALID_ARG for a bad row range.
 */
VS_API vs_status vs_sparse_attn_fwd_rows(const vs_params* p, const vs_index* index, const void* Q, const void* K,
                                         const void* V, void* O, float* lse, void* ws, size_t ws_bytes,
                                         int32_t row_lo, int32_t row_hi, void* stream);

/*
 * Backward of vs_sparse_attn_fwd with the mask held fixed:
 * dV = P^T dO, dS = P * (dO V^T - rowsum(dO * O)), dQ = scale dS K,
 * dK = scale dS^T Q; dK and dV sum over the Hq/Hkv query heads sharing a
 * key/value head and are written (not accumulated).
 *
 * Workspace: at least vs_workspace_bytes(p, VS_OP_BWD_MIN) bytes, else
 * VS_ERR_WORKSPACE.  Bytes beyond that hold the dS tiles (bf16, 2 bytes per
 * active 64 x 64 block entry): the dK / dV pass stores every active block it
 * forms and dQ is computed from them, without forming S and dP a second
 * time.  When the room cannot hold every head's expected blocks (a
 * budget-fill index of density p->density: 1.5x its share of the causal
 * blocks, 2x with index_mode 1, plus four vertical chunks per query block),
 * the call runs in passes over whole key/value head groups, as few as give
 * each head that room; the blocks of one pass are stored and read back
 * before the next reuses the room.  For top-p selection (density 0) it runs
 * one pass.  If the index needs more blocks per head than the room gives
 * (decided on the device, per call), dQ recomputes them instead; the
 * results agree within the stated tolerance either way (and are the same
 * bits for any number of passes).  vs_workspace_bytes(p, VS_OP_BWD) suggests
 * room for the expected blocks of every head in one pass up to 32 GiB, else
 * for the fewest passes whose blocks take at most 96 GiB, else the minimum.
 */
VS_API vs_status vs_sparse_attn_bwd(const vs_params* p, const vs_index* index, const void* Q, const void* K,
                             const void* V, const void* O, const float* lse, const void* dO, void* dQ,
                             void* dK, void* dV, void* ws, size_t ws_bytes, void* stream);

/*
 * Striped sparse ring attention, forward ("平衡稀疏环注意力" section: W =
 * p->stripes workers, token t on worker t mod W at local position t div W;
 * ring-attention page, sections 2.1 and 3.1).  The W workers' ring is run
 * step by step on this GPU: worker r, at step t, attends its queries to KV
 * shard s = (r - t) mod W under the shared index (slash bands in the
 * shard-local 64 x 64 tiles, i.e. the index vs_index_build builds with the
 * same p->stripes; verticals as global tokens) and the local causal rule
 * (key j <= query i when s <= r, j < i when s > r), and folds the step into
 * a carried fp32 (output, log-sum-exp) state.  The result equals
 * vs_sparse_attn_fwd on the same index up to rounding.  Steps run worker by
 * worker (r = 0..W-1, t = 0..W-1).
 *   step_events: optional array of n_events cudaEvent_t (passed as void*),
 *   created by the caller; event r * W + t is recorded on `stream` before
 *   step (r, t) and event W * W after the last step, so that
 *   cudaEventElapsedTime gives each step's time.  NULL / 0: no events;
 *   events beyond n_events are not recorded.
 * Layouts, ownership and errors as vs_sparse_attn_fwd; ws of
 * vs_workspace_bytes(p, VS_OP_RING_FWD) bytes.
 */
VS_API vs_status vs_striped_ring_fwd(const vs_params* p, const vs_index* index, const void* Q, const void* K,
                                     const void* V, void* O, float* lse, void* ws, size_t ws_bytes,
                                     void* const* step_events, int32_t n_events, void* stream);

/*
 * Backward of the striped sparse ring (same ring order): with the final O
 * and lse of every query, each step (r, t) adds its exact share of dQ of
 * worker r (summed in fp32 across the worker's steps) and of dK, dV of shard
 * s (summed in fp32 across workers), written as bf16 at the end.  Equals
 * vs_sparse_attn_bwd on the same index up to rounding.  d = 128 only
 * (VS_ERR_UNSUPPORTED otherwise).  Events, layouts and errors as
 * vs_striped_ring_fwd; ws of vs_workspace_bytes(p, VS_OP_RING_BWD) bytes.
 */
VS_API vs_status vs_striped_ring_bwd(const vs_params* p, const vs_index* index, const void* Q, const void* K,
                                     const void* V, const void* O, const float* lse, const void* dO, void* dQ,
                                     void* dK, void* dV, void* ws, size_t ws_bytes, void* const* step_events,
                                     int32_t n_events, void* stream);

/*
 * Reads the device-side status word of workspace `ws` (synchronises
 * `stream` first) and clears it.  Returns VS_OK, VS_ERR_TIMEOUT, or (in a
 * library built with VS_DEBUG, whose kernels check their global-memory
 * indices, record the first failure and skip the access) VS_ERR_BOUNDS.
 */
VS_API vs_status vs_device_status(void* ws, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* VS_H_ */
