// runtime.cu - the DFlash drafter context behind the C ABI of dflash.h:
// validation, the paged KV pool and its host-side page allocator, the RoPE
// table, TMA descriptors, workspaces, and the call sequences of
// dflash_fuse_ctx / dflash_draft / dflash_verify.
//
// Host/device split of the sequence state: the device holds the exact
// committed length (verify commits on the device, so no call has to wait for
// it); the host holds the pending count exactly and an upper bound of the
// committed length, which sizes page reservations and launch grids. The
// bound is tightened from an asynchronous snapshot of the device lengths
// taken after each verify, once that copy has landed.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <map>
#include <memory>
#include <queue>
#include <string>
#include <tuple>
#include <vector>

#include "dflash.h"
#include "internal.h"
#include <nvtx3/nvToolsExt.h>

using namespace dfl;

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::string g_create_error = "no error";

bool load_encode() {
  if (g_encode) return true;
  cudaDriverEntryPointQueryResult q;
  void* fn = nullptr;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return false;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return true;
}

// Row-major [rows, cols] bf16 matrix, box = 64 columns x box_rows rows, 128B swizzle.
bool encode_2d(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [rows][heads][d] bf16, box = 64 dims x 1 head x box_rows rows.
bool encode_3d(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t heads, uint64_t d, uint32_t box_rows) {
  cuuint64_t dims[3] = {d, heads, rows};
  cuuint64_t strides[2] = {d * 2, heads * d * 2};
  cuuint32_t box[3] = {64, 1, box_rows};
  cuuint32_t es[3] = {1, 1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

}  // namespace

namespace dfl {
// Descriptor helpers and the context-free error string, for entry points
// defined in other translation units.
bool encode_matrix_map(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  return load_encode() && encode_2d(m, ptr, rows, cols, box_rows);
}
void set_unattached_error(const char* msg) { g_create_error = msg; }
}  // namespace dfl

struct dflash_ctx {
  dflash_config cfg{};
  dflash_weights w{};
  std::vector<dflash_layer_weights> layers;
  int num_sms = 0;
  int pages_per_seq = 0;
  int rope_positions = 0;

  // device memory
  uint16_t* pool = nullptr;
  float2* rope = nullptr;
  int* d_len = nullptr;
  int* d_pend = nullptr;
  int* d_page_table = nullptr;
  int* d_status = nullptr;
  float* x = nullptr;        // [max_rows, H] residual stream (fp32)
  uint16_t* hg = nullptr;    // [max_rows, H] bf16(x * gain of the next RMSNorm)
  float* ssA = nullptr;      // [parts][max_rows] partial sums of x^2 (embed / down producers)
  float* ssB = nullptr;      // [parts][max_rows] partial sums of x^2 (O producer)
  uint16_t* q = nullptr;     // [max_rows, n_q*d]
  uint16_t* kb = nullptr;    // [max_rows, n_kv*d] block keys
  uint16_t* vb = nullptr;    // [max_batch][n_kv][d][64 slots] block values, transposed
  uint16_t* attn = nullptr;  // [max_rows, n_q*d]
  uint16_t* act = nullptr;   // [max_rows, F]
  uint16_t* htg = nullptr;   // [max_fuse_tokens, H] bf16(W_c X * g_c)
  float* ssF = nullptr;      // [parts][max_fuse_tokens] partial sums of (W_c X)^2
  float* part_o = nullptr;
  float2* part_ml = nullptr;
  int items_cap = 0;
  float* split_ws = nullptr;
  size_t split_elems = 0;
  int* tickets = nullptr;
  int n_tickets = 0;
  unsigned long long* keys = nullptr;
  int* done = nullptr;
  float* top_logit = nullptr;

  // path selector (installed by dflash_set_path_selector)
  bool sel_on = false;
  CUtensorMap m_wh{};
  float* sel_table = nullptr;              // [V][512] W_A E | W_B E
  float* sel_logits = nullptr;             // [max_rows][sel_ld] logits | H
  int sel_ld = 0, sel_hcol = 0;
  unsigned long long* sel_part = nullptr;  // [max_rows][32][16] slice keys
  float* sel_scores = nullptr;             // [max_rows][16][16]
  int32_t* sel_cand = nullptr;             // [max_rows][16]
  float* sel_cand_u = nullptr;             // [max_rows][16]
  int32_t* sel_next = nullptr;             // [max_rows][16]
  unsigned long long* samp_part = nullptr; // [max_rows][64][32] sampling slice lists
  int* sel_tickets = nullptr;              // [max_batch]

  // two-tap convolutions (installed by dflash_set_conv)
  bool conv_on = false;
  int conv_rank = 0, conv_alloc_rank = 0;
  std::vector<dflash_conv_site> conv_sites;   // [n_layers][ai, ao, fi, fo]
  uint16_t* conv_fold = nullptr;   // per layer: V_ao W_o [2r][n_q d], then V_fo W_d [2r][F]
  uint16_t* conv_vt = nullptr;     // per layer: V_ai^T, then V_fi^T, each [H][2r]
  float* conv_yp = nullptr;        // [max_rows][H + 2r] sublayer output | its products with V
  uint16_t* conv_h = nullptr;      // [max_rows][H] convolved input of QKV / gate-up
  float* conv_p = nullptr;         // [max_rows][2r] layer 0's V_ai products (scaled)
  float* conv_acc = nullptr;       // [2][max_rows][2r] accumulators of an input site's products
  std::vector<CUtensorMap> m_fold_o, m_fold_d;
  CUtensorMap m_vai0{};

  // weight descriptors
  std::vector<CUtensorMap> m_wq, m_wk, m_wv, m_wo, m_wg, m_wu, m_wd;
  CUtensorMap m_lm{}, m_wc{}, m_pool{}, m_pool_vt{}, m_vblk{};
  std::map<std::tuple<const void*, int, int, int, int>, CUtensorMap> act_maps;

  // host view of the sequences
  std::vector<int> free_pages;
  std::vector<std::vector<int>> pages;
  std::vector<int> len_ub, pend, added_since;
  int* h_snap = nullptr;      // pinned copy of d_len
  std::vector<double> deal_load;   // scratch of the attention work split
  std::vector<std::pair<int, uint32_t>> deal_items;
  std::vector<int> deal_owner, deal_count;
  std::unique_ptr<AttnSched> attn_sched{new AttnSched()};
  std::unique_ptr<PageUpdates> page_upd{new PageUpdates()};   // staging of one append's new pages
  cudaEvent_t snap_event = nullptr;
  bool snap_pending = false;

  // target mode (dflash_target_create): a causal pass over caller ids that
  // caches its own K/V; feat_slot[l] = index of layer l among the feature
  // layers, or -1
  bool target = false;
  std::vector<int> feat_slot;
  int n_feat = 0;

  int last_rows = 0, last_draft_rows = 0, last_sel_rows = 0;
  int attn_ctas_per_sm = 0;
  std::string err = "no error";

  // per-kernel accounting
  bool prof_on = false;
  std::vector<cudaEvent_t> prof_events;
  size_t prof_next = 0;
  std::vector<std::pair<int, size_t>> prof_recs;   // (class, first event)
  dflash_kernel_stat prof_acc[DFLASH_K_COUNT] = {};

  int max_rows() const { return cfg.max_batch * cfg.max_block; }
};

namespace {

// One NVTX range per API call (header-only NVTX 3: a no-op unless a profiler
// is attached).
struct ApiRange {
  explicit ApiRange(const char* name) { nvtxRangePushA(name); }
  ~ApiRange() { nvtxRangePop(); }
};

dflash_status fail(dflash_ctx* c, dflash_status s, const std::string& msg) {
  if (c) c->err = msg;
  else g_create_error = msg;
  return s;
}

#define CK(call)                                                                                   \
  do {                                                                                             \
    cudaError_t e_ = (call);                                                                       \
    if (e_ != cudaSuccess) return fail(ctx, DFLASH_ECUDA, std::string(#call) + ": " + cudaGetErrorString(e_)); \
  } while (0)

template <typename T>
cudaError_t dalloc(T** p, size_t count) {
  return cudaMalloc(reinterpret_cast<void**>(p), std::max<size_t>(count, 1) * sizeof(T));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

const CUtensorMap* act_map(dflash_ctx* ctx, const void* ptr, int rows, int cols, int box_rows) {
  auto key = std::make_tuple(ptr, rows, cols, box_rows, 2);
  auto it = ctx->act_maps.find(key);
  if (it != ctx->act_maps.end()) return &it->second;
  CUtensorMap m;
  if (!encode_2d(&m, ptr, rows, cols, box_rows)) return nullptr;
  if (ctx->act_maps.size() > 4096) ctx->act_maps.clear();
  return &(ctx->act_maps[key] = m);
}

// The block's queries [rows][n_q][d], box = 64 dims x G heads x B rows: the
// G*B query rows of one (sequence, kv head) in one copy.
const CUtensorMap* blk_map(dflash_ctx* ctx, const void* ptr, int rows, int box_rows) {
  auto key = std::make_tuple(ptr, rows, ctx->cfg.n_kv_heads, box_rows, 3);
  auto it = ctx->act_maps.find(key);
  if (it != ctx->act_maps.end()) return &it->second;
  CUtensorMap m;
  if (!encode_3d(&m, ptr, rows, ctx->cfg.n_kv_heads, ctx->cfg.head_dim, box_rows)) return nullptr;
  return &(ctx->act_maps[key] = m);
}

// Counts one launch group of class `cls` with its algorithmic bytes/flops and,
// while profiling is on, brackets it with events on the launch stream.
struct ProfScope {
  dflash_ctx* c;
  int cls;
  cudaStream_t s;
  size_t ev = static_cast<size_t>(-1);
  ProfScope(dflash_ctx* c_, int cls_, cudaStream_t s_, double bytes, double flops, int launches = 1)
      : c(c_), cls(cls_), s(s_) {
    c->prof_acc[cls].launches += launches;
    c->prof_acc[cls].bytes += bytes;
    c->prof_acc[cls].flops += flops;
    if (!c->prof_on) return;
    while (c->prof_next + 2 > c->prof_events.size()) {
      cudaEvent_t e;
      if (cudaEventCreate(&e) != cudaSuccess) return;
      c->prof_events.push_back(e);
    }
    ev = c->prof_next;
    c->prof_next += 2;
    cudaEventRecord(c->prof_events[ev], s);
  }
  ~ProfScope() {
    if (ev == static_cast<size_t>(-1)) return;
    cudaEventRecord(c->prof_events[ev + 1], s);
    c->prof_recs.emplace_back(cls, ev);
  }
};

// Algorithmic traffic of OUT[M, n_out] = X[M, K] W[n_w, K]^T with `ob` bytes
// per output element (read-modify-write outputs count twice).
double gemm_bytes(double M, double n_w, double K, double n_out, double ob) {
  return n_w * K * 2 + M * K * 2 + M * n_out * ob;
}

SeqState seq_state(dflash_ctx* ctx) {
  SeqState s;
  s.len = ctx->d_len;
  s.pend = ctx->d_pend;
  s.page_table = ctx->d_page_table;
  s.pages_per_seq = ctx->pages_per_seq;
  return s;
}

GemmWork gemm_work(dflash_ctx* ctx) {
  GemmWork w;
  w.partial = ctx->split_ws;
  w.partial_elems = ctx->split_elems;
  w.tickets = ctx->tickets;
  w.n_tickets = ctx->n_tickets;
  return w;
}

GemmEpi base_epi(dflash_ctx* ctx, int kind) {
  GemmEpi e;
  std::memset(&e, 0, sizeof(e));
  e.kind = kind;
  e.head_dim = ctx->cfg.head_dim;
  e.n_q_heads = ctx->cfg.n_heads;
  e.n_kv_heads = ctx->cfg.n_kv_heads;
  e.rope = ctx->rope;
  e.rope_positions = ctx->rope_positions;
  e.seqs = seq_state(ctx);
  e.pool = ctx->pool;
  e.pool_pages = ctx->cfg.max_pages;
  e.kv_q8 = ctx->cfg.kv_format == 1;
  e.status = ctx->d_status;
  e.inv_hidden = 1.0f / ctx->cfg.hidden;
  e.eps = ctx->cfg.rms_eps;
  return e;
}

ARegions stacked(std::initializer_list<int> rows) {
  ARegions r;
  std::memset(&r, 0, sizeof(r));
  int t = 0, i = 0;
  for (int n : rows) {
    r.tile_begin[i++] = t;
    t += ceil_div(n, 128);
  }
  r.tile_begin[i] = t;
  r.n_regions = i;
  r.paired = 0;
  r.pair = 64;
  return r;
}

void release_tail_pages(dflash_ctx* ctx, int s) {
  const int need = ceil_div(ctx->len_ub[s] + ctx->pend[s], kPage);
  auto& pg = ctx->pages[s];
  while (static_cast<int>(pg.size()) > need) {
    ctx->free_pages.push_back(pg.back());
    pg.pop_back();
  }
}

// Tighten the host's committed-length bounds from a landed snapshot.
void consume_snapshot(dflash_ctx* ctx, bool force_wait) {
  if (!ctx->snap_pending) return;
  if (force_wait) cudaEventSynchronize(ctx->snap_event);
  else if (cudaEventQuery(ctx->snap_event) != cudaSuccess) return;
  for (int s = 0; s < ctx->cfg.max_seqs; ++s) {
    const int exact = ctx->h_snap[s] + ctx->added_since[s];
    if (exact < ctx->len_ub[s]) {
      ctx->len_ub[s] = exact;
      release_tail_pages(ctx, s);
    }
    ctx->added_since[s] = 0;
  }
  ctx->snap_pending = false;
}

dflash_status check_seqs(dflash_ctx* ctx, const int32_t* seq_ids, int n_seq, SeqMeta* meta) {
  if (n_seq < 0 || n_seq > ctx->cfg.max_batch) return fail(ctx, DFLASH_EINVAL, "n_seq out of range");
  if (n_seq > 0 && !seq_ids) return fail(ctx, DFLASH_EINVAL, "seq_ids is null");
  std::memset(meta, 0, sizeof(*meta));
  meta->n_seq = n_seq;
  for (int i = 0; i < n_seq; ++i) {
    const int s = seq_ids[i];
    if (s < 0 || s >= ctx->cfg.max_seqs) return fail(ctx, DFLASH_EINVAL, "sequence id out of range");
    for (int j = 0; j < i; ++j)
      if (seq_ids[j] == s) return fail(ctx, DFLASH_EINVAL, "duplicate sequence id in one call");
    meta->slot[i] = s;
  }
  return DFLASH_OK;
}

}  // namespace

extern "C" {

const char* dflash_last_error(const dflash_ctx* ctx) { return ctx ? ctx->err.c_str() : g_create_error.c_str(); }

dflash_status dflash_destroy(dflash_ctx* ctx) {
  if (!ctx) return DFLASH_EINVAL;
  cudaDeviceSynchronize();
  void* ptrs[] = {ctx->pool, ctx->rope, ctx->d_len, ctx->d_pend, ctx->d_page_table, ctx->d_status, ctx->x,
                  ctx->hg, ctx->ssA, ctx->ssB, ctx->q, ctx->kb, ctx->vb, ctx->attn, ctx->act, ctx->htg, ctx->ssF,
                  ctx->part_o, ctx->part_ml, ctx->split_ws, ctx->tickets, ctx->keys, ctx->done, ctx->top_logit,
                  ctx->sel_table, ctx->sel_logits, ctx->sel_part, ctx->sel_scores, ctx->sel_cand, ctx->sel_cand_u,
                  ctx->sel_tickets, ctx->sel_next,
                  ctx->samp_part, ctx->conv_fold, ctx->conv_vt, ctx->conv_yp, ctx->conv_h, ctx->conv_p,
                  ctx->conv_acc};
  for (void* p : ptrs)
    if (p) cudaFree(p);
  if (ctx->h_snap) cudaFreeHost(ctx->h_snap);
  for (cudaEvent_t e : ctx->prof_events) cudaEventDestroy(e);
  if (ctx->snap_event) cudaEventDestroy(ctx->snap_event);
  delete ctx;
  return DFLASH_OK;
}

}  // extern "C"

namespace {

// feat_layers == nullptr: a drafter context; otherwise a target context whose
// cfg->n_feat_layers feature layers are feat_layers[0 ..] (0-based, strictly
// increasing); the fusion weights are not used.
dflash_status create_impl(const dflash_config* cfg_in, const dflash_weights* w, const int32_t* feat_layers,
                          dflash_ctx** out) {
  dflash_ctx* ctx = nullptr;
  if (!out) return fail(nullptr, DFLASH_EINVAL, "out is null");
  *out = nullptr;
  if (!cfg_in || !w || !w->layers) return fail(nullptr, DFLASH_EINVAL, "null config or weights");
  dflash_config c = *cfg_in;
  const bool target = feat_layers != nullptr;
  if (target) c.max_fuse_tokens = 1;   // no fusion in a target context
  const int d = c.head_dim;
  if (c.hidden < 64 || c.hidden % 64) return fail(nullptr, DFLASH_EINVAL, "hidden must be a positive multiple of 64");
  if (d != 64 && d != 128) return fail(nullptr, DFLASH_EINVAL, "head_dim must be 64 or 128");
  if (c.n_kv_heads < 1 || c.n_heads < 1 || c.n_heads % c.n_kv_heads)
    return fail(nullptr, DFLASH_EINVAL, "n_heads must be a multiple of n_kv_heads");
  if ((c.n_heads * d) % 128 || (c.n_kv_heads * d) % 128)
    return fail(nullptr, DFLASH_EINVAL, "n_heads*d and n_kv_heads*d must be multiples of 128");
  if (c.ffn < 8 || c.ffn % 8) return fail(nullptr, DFLASH_EINVAL, "ffn must be a positive multiple of 8");
  if (c.vocab < 2 || c.mask_id < 0 || c.mask_id >= c.vocab) return fail(nullptr, DFLASH_EINVAL, "bad vocab/mask_id");
  if (!target && (c.n_layers < 1 || c.n_layers > 16 || c.n_feat_layers < 1 || c.n_feat_layers > 16))
    return fail(nullptr, DFLASH_EINVAL, "n_layers and n_feat_layers must be in 1..16");
  if (target) {
    if (c.n_layers < 1 || c.n_layers > kMaxTargetLayers || c.n_feat_layers < 0 || c.n_feat_layers > 16)
      return fail(nullptr, DFLASH_EINVAL, "target: n_layers must be in 1..64 and n_feat_layers in 0..16");
    for (int k = 0; k < c.n_feat_layers; ++k)
      if (feat_layers[k] < 0 || feat_layers[k] >= c.n_layers || (k > 0 && feat_layers[k] <= feat_layers[k - 1]))
        return fail(nullptr, DFLASH_EINVAL, "target: feature layers must be increasing layer indices");
  }
  if (c.max_batch < 1 || c.max_batch > kMaxBatch) return fail(nullptr, DFLASH_EINVAL, "max_batch must be in 1..64");
  if (c.max_block < 1 || c.max_block > kMaxBlock) return fail(nullptr, DFLASH_EINVAL, "max_block must be in 1..32");
  if ((c.n_heads / c.n_kv_heads) * c.max_block > 128)
    return fail(nullptr, DFLASH_EINVAL, "(n_heads/n_kv_heads)*max_block must be at most 128");
  if (c.max_seqs < 1 || c.max_ctx < 1 || c.max_pages < 1 || c.max_fuse_tokens < 1)
    return fail(nullptr, DFLASH_EINVAL, "capacities must be positive");
  if (!(c.rms_eps >= 0.f) || !(c.rope_base > 1.f)) return fail(nullptr, DFLASH_EINVAL, "bad rms_eps or rope_base");
  if (c.kv_format != 0 && c.kv_format != 1) return fail(nullptr, DFLASH_EINVAL, "kv_format must be 0 or 1");
  if (c.kv_format == 1 && target) return fail(nullptr, DFLASH_EINVAL, "8-bit K/V pages are for drafter contexts");
  const bool q8 = c.kv_format == 1;
  const long long pool_rows = 1LL * c.n_layers * c.max_pages * 2 * c.n_kv_heads * kPage;
  // the pool is also read as rows of 64 elements (transposed values)
  if (!q8 && pool_rows * (d / 64) >= (1LL << 31))
    return fail(nullptr, DFLASH_EINVAL, "KV pool too large for 32-bit TMA coordinates");
  // 8-bit pages: 136 d bytes per (layer, page, kv head), held as 16-bit elements
  const size_t pool_elems = q8 ? 1ull * c.n_layers * c.max_pages * c.n_kv_heads * q8_head_bytes(d) / 2
                               : static_cast<size_t>(pool_rows) * d;
  const void* ptrs[] = {w->embed, w->lm_head, w->g_final, target ? w->embed : w->w_c, target ? w->embed : w->g_c};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return fail(nullptr, DFLASH_EINVAL, "weight pointer null or not 16-byte aligned");
  for (int l = 0; l < c.n_layers; ++l) {
    const dflash_layer_weights& L = w->layers[l];
    const void* lp[] = {L.w_q, L.w_k, L.w_v, L.w_o, L.w_gate, L.w_up, L.w_down, L.g_attn, L.g_ffn};
    for (const void* p : lp)
      if (!p || !aligned16(p)) return fail(nullptr, DFLASH_EINVAL, "layer weight null or not 16-byte aligned");
  }
  if (!load_encode()) return fail(nullptr, DFLASH_ECUDA, "cuTensorMapEncodeTiled unavailable");

  ctx = new dflash_ctx();
  ctx->cfg = c;
  ctx->target = target;
  ctx->feat_slot.assign(c.n_layers, -1);
  if (target) {
    ctx->n_feat = c.n_feat_layers;
    for (int k = 0; k < c.n_feat_layers; ++k) ctx->feat_slot[feat_layers[k]] = k;
  }
  ctx->layers.assign(w->layers, w->layers + c.n_layers);
  ctx->w = *w;
  ctx->w.layers = ctx->layers.data();
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&ctx->num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) {
    g_create_error = std::string("no CUDA device: ") + cudaGetErrorString(e);
    delete ctx;
    return DFLASH_ECUDA;
  }
  const int H = c.hidden, nq = c.n_heads, nkv = c.n_kv_heads, F = c.ffn;
  ctx->pages_per_seq = ceil_div(c.max_ctx, kPage);
  ctx->rope_positions = c.max_ctx + c.max_block;
  const size_t rows = ctx->max_rows();
  const int G = nq / nkv;
  const int rows_pad = 16 * ceil_div(G * c.max_block, 16);
  ctx->items_cap = 4 * ctx->num_sms + c.max_batch * nkv + 64;

  auto bad = [&](cudaError_t err, const char* what) {
    g_create_error = std::string(what) + ": " + cudaGetErrorString(err);
    dflash_destroy(ctx);
    return err == cudaErrorMemoryAllocation ? DFLASH_ENOMEM : DFLASH_ECUDA;
  };
#define CA(call, what)                      \
  do {                                      \
    cudaError_t e_ = (call);                \
    if (e_ != cudaSuccess) return bad(e_, what); \
  } while (0)

  CA(dalloc(&ctx->pool, pool_elems), "KV pool");
  CA(cudaMemset(ctx->pool, 0, pool_elems * 2), "KV pool");
  CA(dalloc(&ctx->rope, static_cast<size_t>(ctx->rope_positions) * (d / 2)), "RoPE table");
  CA(dalloc(&ctx->d_len, c.max_seqs), "lengths");
  CA(dalloc(&ctx->d_pend, c.max_seqs), "lengths");
  CA(cudaMemset(ctx->d_len, 0, c.max_seqs * sizeof(int)), "lengths");
  CA(cudaMemset(ctx->d_pend, 0, c.max_seqs * sizeof(int)), "lengths");
  CA(dalloc(&ctx->d_page_table, static_cast<size_t>(c.max_seqs) * ctx->pages_per_seq), "page table");
  CA(cudaMemset(ctx->d_page_table, 0xFF, static_cast<size_t>(c.max_seqs) * ctx->pages_per_seq * sizeof(int)),
     "page table");
  CA(dalloc(&ctx->d_status, 1), "status");
  CA(cudaMemset(ctx->d_status, 0, sizeof(int)), "status");
  const int parts = ceil_div(H, 128);
  CA(dalloc(&ctx->x, rows * H), "workspace");
  CA(dalloc(&ctx->hg, rows * H), "workspace");
  // sums-of-squares parts: 128-column GEMM tiles, or the convolutions' 32-column parts
  CA(dalloc(&ctx->ssA, rows * ceil_div(H, kConvCols)), "workspace");
  CA(dalloc(&ctx->ssB, rows * ceil_div(H, kConvCols)), "workspace");
  CA(dalloc(&ctx->q, rows * nq * d), "workspace");
  CA(dalloc(&ctx->kb, rows * nkv * d), "workspace");
  const size_t vb_elems = static_cast<size_t>(c.max_batch) * nkv * d * kPage;
  CA(dalloc(&ctx->vb, vb_elems), "workspace");
  CA(cudaMemset(ctx->kb, 0, rows * nkv * d * 2), "workspace");
  CA(cudaMemset(ctx->vb, 0, vb_elems * 2), "workspace");
  CA(dalloc(&ctx->attn, rows * nq * d), "workspace");
  CA(dalloc(&ctx->act, rows * F), "workspace");
  CA(dalloc(&ctx->htg, static_cast<size_t>(c.max_fuse_tokens) * H), "workspace");
  CA(dalloc(&ctx->ssF, static_cast<size_t>(c.max_fuse_tokens) * parts), "workspace");
  CA(dalloc(&ctx->part_o, static_cast<size_t>(ctx->items_cap) * rows_pad * d), "attention partials");
  CA(dalloc(&ctx->part_ml, static_cast<size_t>(ctx->items_cap) * rows_pad), "attention partials");
  ctx->split_elems = static_cast<size_t>(16) << 20;   // 2 slots of 128 x 256 floats for 256 CTAs
  CA(dalloc(&ctx->split_ws, ctx->split_elems), "split-K workspace");
  ctx->n_tickets = 1 << 16;
  CA(dalloc(&ctx->tickets, ctx->n_tickets), "tickets");
  CA(cudaMemset(ctx->tickets, 0, ctx->n_tickets * sizeof(int)), "tickets");
  CA(dalloc(&ctx->keys, rows), "argmax keys");
  CA(cudaMemset(ctx->keys, 0, rows * sizeof(unsigned long long)), "argmax keys");
  CA(dalloc(&ctx->done, 1), "argmax counter");
  CA(cudaMemset(ctx->done, 0, sizeof(int)), "argmax counter");
  CA(dalloc(&ctx->top_logit, rows), "top logits");
  CA(cudaMallocHost(reinterpret_cast<void**>(&ctx->h_snap), c.max_seqs * sizeof(int)), "pinned snapshot");
  CA(cudaEventCreateWithFlags(&ctx->snap_event, cudaEventDisableTiming), "event");

  // RoPE table: angle pos * base^(-2i/d) in double precision, stored as fp32 (cos, sin).
  {
    std::vector<float2> tab(static_cast<size_t>(ctx->rope_positions) * (d / 2));
    for (int i = 0; i < d / 2; ++i) {
      const double theta = std::pow(static_cast<double>(c.rope_base), -2.0 * i / d);
      for (int p = 0; p < ctx->rope_positions; ++p) {
        const double a = p * theta;
        tab[static_cast<size_t>(p) * (d / 2) + i] = make_float2(static_cast<float>(std::cos(a)), static_cast<float>(std::sin(a)));
      }
    }
    CA(cudaMemcpy(ctx->rope, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice), "RoPE table");
  }

  // weight descriptors (box 64 K-elements x 64 rows)
  const int wb = kWeightBoxRows;
  bool ok = encode_2d(&ctx->m_lm, w->lm_head, c.vocab, H, wb) &&
            (target || encode_2d(&ctx->m_wc, w->w_c, H, static_cast<uint64_t>(c.n_feat_layers) * H, wb)) &&
            (q8 || encode_2d(&ctx->m_pool, ctx->pool, pool_rows, d, 64)) &&
            (q8 || encode_2d(&ctx->m_pool_vt, ctx->pool, static_cast<uint64_t>(pool_rows) * (d / 64), 64, 64)) &&
            encode_2d(&ctx->m_vblk, ctx->vb, static_cast<uint64_t>(c.max_batch) * nkv * d, 64, 64);
  ctx->m_wq.resize(c.n_layers);
  ctx->m_wk.resize(c.n_layers);
  ctx->m_wv.resize(c.n_layers);
  ctx->m_wo.resize(c.n_layers);
  ctx->m_wg.resize(c.n_layers);
  ctx->m_wu.resize(c.n_layers);
  ctx->m_wd.resize(c.n_layers);
  for (int l = 0; l < c.n_layers && ok; ++l) {
    const dflash_layer_weights& L = ctx->layers[l];
    ok = encode_2d(&ctx->m_wq[l], L.w_q, nq * d, H, wb) && encode_2d(&ctx->m_wk[l], L.w_k, nkv * d, H, wb) &&
         encode_2d(&ctx->m_wv[l], L.w_v, nkv * d, H, wb) && encode_2d(&ctx->m_wo[l], L.w_o, H, nq * d, wb) &&
         encode_2d(&ctx->m_wg[l], L.w_gate, F, H, wb) && encode_2d(&ctx->m_wu[l], L.w_up, F, H, wb) &&
         encode_2d(&ctx->m_wd[l], L.w_down, H, F, wb);
  }
  if (!ok) {
    g_create_error = "cuTensorMapEncodeTiled rejected a weight layout";
    dflash_destroy(ctx);
    return DFLASH_EINVAL;
  }
  CA(cudaDeviceSynchronize(), "create");

  ctx->free_pages.reserve(c.max_pages);
  for (int p = c.max_pages - 1; p >= 0; --p) ctx->free_pages.push_back(p);
  ctx->pages.assign(c.max_seqs, {});
  ctx->len_ub.assign(c.max_seqs, 0);
  ctx->pend.assign(c.max_seqs, 0);
  ctx->added_since.assign(c.max_seqs, 0);
  *out = ctx;
#undef CA
  return DFLASH_OK;
}

}  // namespace

extern "C" {

dflash_status dflash_create(const dflash_config* cfg, const dflash_weights* w, dflash_ctx** out) {
  return create_impl(cfg, w, nullptr, out);
}

dflash_status dflash_target_create(const dflash_config* cfg, const dflash_weights* w, const int32_t* feat_layers,
                                   dflash_ctx** out) {
  static const int32_t none = 0;
  if (cfg && cfg->n_feat_layers > 0 && !feat_layers) return fail(nullptr, DFLASH_EINVAL, "feat_layers is null");
  return create_impl(cfg, w, feat_layers ? feat_layers : &none, out);
}

dflash_status dflash_target_feature_layers(int n_layers, int n_feat, int32_t* out) {
  if (n_layers < 5 || n_feat < 1 || n_feat > 16 || !out || n_feat > n_layers - 3) return DFLASH_EINVAL;
  // uniformly spaced from layer 2 to the third-to-last (1-based), to the nearest layer
  const int first = 2, last = n_layers - 2;
  for (int k = 0; k < n_feat; ++k) {
    const double pos = n_feat == 1 ? first : first + k * static_cast<double>(last - first) / (n_feat - 1);
    out[k] = static_cast<int32_t>(std::floor(pos + 0.5)) - 1;
  }
  return DFLASH_OK;
}

dflash_status dflash_sync(dflash_ctx* ctx) {
  if (!ctx) return DFLASH_EINVAL;
  CK(cudaDeviceSynchronize());
  int st = 0;
  CK(cudaMemcpy(&st, ctx->d_status, sizeof(int), cudaMemcpyDeviceToHost));
  if (st) {
    CK(cudaMemset(ctx->d_status, 0, sizeof(int)));
    if (st & kDevTimeout) return fail(ctx, DFLASH_ETIMEOUT, "a kernel's bounded wait ran out");
    return fail(ctx, DFLASH_EDEVICE, "a kernel found an index out of range");
  }
  return DFLASH_OK;
}

dflash_status dflash_seq_reset(dflash_ctx* ctx, int seq) {
  if (!ctx) return DFLASH_EINVAL;
  if (seq < 0 || seq >= ctx->cfg.max_seqs) return fail(ctx, DFLASH_EINVAL, "sequence id out of range");
  CK(cudaDeviceSynchronize());
  consume_snapshot(ctx, true);
  CK(cudaMemset(ctx->d_len + seq, 0, sizeof(int)));
  CK(cudaMemset(ctx->d_pend + seq, 0, sizeof(int)));
  ctx->len_ub[seq] = 0;
  ctx->pend[seq] = 0;
  ctx->added_since[seq] = 0;
  release_tail_pages(ctx, seq);
  return DFLASH_OK;
}

dflash_status dflash_seq_len(dflash_ctx* ctx, int seq, int* committed, int* pending) {
  if (!ctx) return DFLASH_EINVAL;
  if (seq < 0 || seq >= ctx->cfg.max_seqs) return fail(ctx, DFLASH_EINVAL, "sequence id out of range");
  CK(cudaDeviceSynchronize());
  consume_snapshot(ctx, true);
  std::vector<int> lens(ctx->cfg.max_seqs);
  CK(cudaMemcpy(lens.data(), ctx->d_len, lens.size() * sizeof(int), cudaMemcpyDeviceToHost));
  int p = 0;
  CK(cudaMemcpy(&p, ctx->d_pend + seq, sizeof(int), cudaMemcpyDeviceToHost));
  for (int s = 0; s < ctx->cfg.max_seqs; ++s) {
    ctx->len_ub[s] = lens[s];
    ctx->added_since[s] = 0;
    release_tail_pages(ctx, s);
  }
  if (committed) *committed = lens[seq];
  if (pending) *pending = p;
  return DFLASH_OK;
}

dflash_status dflash_fuse_ctx(dflash_ctx* ctx, const int32_t* seq_ids, int n_seq, const int32_t* n_new,
                              const uint16_t* feats, int pending, void* stream_v) {
  ApiRange nvtx_range("dflash_fuse_ctx");
  if (!ctx) return DFLASH_EINVAL;
  if (ctx->target) return fail(ctx, DFLASH_EINVAL, "a target context has no fusion (its pass caches its own K/V)");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  const dflash_config& c = ctx->cfg;
  SeqMeta meta;
  dflash_status st = check_seqs(ctx, seq_ids, n_seq, &meta);
  if (st != DFLASH_OK) return st;
  if (n_seq > 0 && !n_new) return fail(ctx, DFLASH_EINVAL, "n_new is null");
  if (pending != 0 && pending != 1) return fail(ctx, DFLASH_EINVAL, "pending must be 0 or 1");
  long long total = 0;
  for (int i = 0; i < n_seq; ++i) {
    if (n_new[i] < 0) return fail(ctx, DFLASH_EINVAL, "n_new must be >= 0");
    meta.row0[i] = static_cast<int>(total);
    total += n_new[i];
  }
  meta.row0[n_seq] = static_cast<int>(total);
  if (total > c.max_fuse_tokens) return fail(ctx, DFLASH_EINVAL, "sum(n_new) exceeds max_fuse_tokens");
  if (total == 0) return DFLASH_OK;
  if (!feats || !aligned16(feats)) return fail(ctx, DFLASH_EINVAL, "feats null or not 16-byte aligned");
  consume_snapshot(ctx, false);
  for (int i = 0; i < n_seq; ++i) {
    const int s = meta.slot[i];
    if (!pending && ctx->pend[s]) return fail(ctx, DFLASH_EINVAL, "committed append while tokens are pending");
    if (ctx->len_ub[s] + ctx->pend[s] + n_new[i] > c.max_ctx) {
      // the bound may be loose: wait for the snapshot before refusing
      consume_snapshot(ctx, true);
      if (ctx->len_ub[s] + ctx->pend[s] + n_new[i] > c.max_ctx)
        return fail(ctx, DFLASH_EINVAL, "append would exceed max_ctx");
    }
  }
  // reserve pages (all or nothing)
  int need_total = 0;
  for (int i = 0; i < n_seq; ++i) {
    const int s = meta.slot[i];
    need_total += std::max(0, ceil_div(ctx->len_ub[s] + ctx->pend[s] + n_new[i], kPage) -
                                  static_cast<int>(ctx->pages[s].size()));
  }
  if (need_total > static_cast<int>(ctx->free_pages.size())) {
    consume_snapshot(ctx, true);
    need_total = 0;
    for (int i = 0; i < n_seq; ++i) {
      const int s = meta.slot[i];
      need_total += std::max(0, ceil_div(ctx->len_ub[s] + ctx->pend[s] + n_new[i], kPage) -
                                    static_cast<int>(ctx->pages[s].size()));
    }
    if (need_total > static_cast<int>(ctx->free_pages.size()))
      return fail(ctx, DFLASH_ENOMEM, "KV page pool exhausted");
  }
  PageUpdates& upd = *ctx->page_upd;
  upd.n = 0;
  for (int i = 0; i < n_seq; ++i) {
    const int s = meta.slot[i];
    auto& pg = ctx->pages[s];
    const int have = static_cast<int>(pg.size());
    const int want = ceil_div(ctx->len_ub[s] + ctx->pend[s] + n_new[i], kPage);
    for (int k = have; k < want; ++k) {
      pg.push_back(ctx->free_pages.back());
      ctx->free_pages.pop_back();
      upd.idx[upd.n] = s * ctx->pages_per_seq + k;
      upd.page[upd.n] = pg.back();
      if (++upd.n == kPageUpdMax) {
        CK(launch_page_updates(upd, ctx->d_page_table, stream));
        upd.n = 0;
      }
    }
  }
  CK(launch_page_updates(upd, ctx->d_page_table, stream));

  const int H = c.hidden, d = c.head_dim, nkv = c.n_kv_heads;
  const int M = static_cast<int>(total);
  GemmWork work = gemm_work(ctx);
  const int parts = ceil_div(H, 128);
  // x = X W_c^T, kept as bf16(x * g_c) plus per-tile sums of x^2: the
  // fusion RMSNorm is applied as a per-token scale by the next GEMM
  {
    AMaps am;
    am.m[0] = ctx->m_wc;
    ARegions rg = stacked({H});
    const CUtensorMap* xm = act_map(ctx, feats, M, c.n_feat_layers * H, gemm_act_rows(M, H, c.n_feat_layers * H, ctx->num_sms));
    if (!xm) return fail(ctx, DFLASH_EINVAL, "cannot describe feats for TMA");
    GemmEpi e = base_epi(ctx, EPI_NORMSRC);
    e.out_hg = ctx->htg;
    e.ld_out = H;
    e.gain = ctx->w.g_c;
    e.out_ss = ctx->ssF;
    e.out_ss_ld = c.max_fuse_tokens;
    const double K = 1.0 * c.n_feat_layers * H;
    ProfScope ps(ctx, DFLASH_K_FUSE_WC, stream, gemm_bytes(M, H, K, H, 2), 2.0 * M * H * K);
    CK(launch_gemm(am, rg, *xm, M, H, c.n_feat_layers * H, 0, e, work, ctx->num_sms, stream));
  }
  // K/V of every layer from H_t = x / rms(x) * g_c, RoPE on K, scattered into the pages
  {
    const int per_launch = kMaxAMaps / 2;
    for (int l0 = 0; l0 < c.n_layers; l0 += per_launch) {
      const int nl = std::min(per_launch, c.n_layers - l0);
      const CUtensorMap* xm =
          act_map(ctx, ctx->htg, M, H, gemm_act_rows(M, 2 * nl * ceil_div(nkv * d, 128) * 128, H, ctx->num_sms));
      if (!xm) return fail(ctx, DFLASH_EINVAL, "cannot describe H_t for TMA");
      AMaps am;
      ARegions rg;
      std::memset(&rg, 0, sizeof(rg));
      const int tiles = ceil_div(nkv * d, 128);
      for (int j = 0; j < nl; ++j) {
        am.m[2 * j] = ctx->m_wk[l0 + j];
        am.m[2 * j + 1] = ctx->m_wv[l0 + j];
        rg.tile_begin[2 * j] = 2 * j * tiles;
        rg.tile_begin[2 * j + 1] = (2 * j + 1) * tiles;
      }
      rg.n_regions = 2 * nl;
      rg.pair = d / 2;
      rg.tile_begin[2 * nl] = 2 * nl * tiles;
      GemmEpi e = base_epi(ctx, EPI_KV_APPEND);
      e.meta = meta;
      e.layer0 = l0;
      e.in_ss = ctx->ssF;
      e.in_ss_parts = parts;
      e.in_ss_ld = c.max_fuse_tokens;
      const double nw = 2.0 * nl * nkv * d;
      const double out_b = c.kv_format == 1 ? 2.125 / 4.0 * 2 : 2;   // bytes per output value
      ProfScope ps(ctx, DFLASH_K_FUSE_KV, stream, gemm_bytes(M, nw, H, nw, out_b), 2.0 * M * nw * H);
      CK(launch_gemm(am, rg, *xm, M, 2 * nl * tiles * 128, H, 0, e, work, ctx->num_sms, stream));
    }
  }
  {
    ProfScope ps(ctx, DFLASH_K_OTHER, stream, 8.0 * n_seq, 0);
    CK(launch_fuse_advance(meta, seq_state(ctx), pending, stream));
  }
  for (int i = 0; i < n_seq; ++i) {
    const int s = meta.slot[i];
    if (pending) ctx->pend[s] += n_new[i];
    else {
      ctx->len_ub[s] += n_new[i];
      ctx->added_since[s] += n_new[i];
    }
  }
  return DFLASH_OK;
}

namespace {

// Temperature-sampling head of a draft (dflash_draft_sample).
struct SampleReq {
  float temperature, top_p;
  int top_k;
  const float* uniforms;
  int32_t* q_ids;
  float* q_probs;
};

// The selector's and the sampling head's fp32 logits rows [max_rows][V_pad + 256]
// and the sampling slice lists, allocated at first use.
dflash_status ensure_logits32(dflash_ctx* ctx) {
  if (ctx->sel_logits) return DFLASH_OK;
  const dflash_config& c = ctx->cfg;
  const size_t rows = ctx->max_rows();
  ctx->sel_hcol = 128 * ceil_div(c.vocab, 128);   // H starts at the first tile after the vocabulary
  ctx->sel_ld = ctx->sel_hcol + kSelDim;
  cudaError_t e = dalloc(&ctx->sel_logits, rows * ctx->sel_ld);
  if (e == cudaSuccess) e = cudaMemset(ctx->sel_logits, 0, rows * ctx->sel_ld * sizeof(float));
  if (e != cudaSuccess) {
    if (ctx->sel_logits) cudaFree(ctx->sel_logits);
    ctx->sel_logits = nullptr;
    return fail(ctx, e == cudaErrorMemoryAllocation ? DFLASH_ENOMEM : DFLASH_ECUDA,
                std::string("logits buffer: ") + cudaGetErrorString(e));
  }
  return DFLASH_OK;
}

dflash_status ensure_sample_part(dflash_ctx* ctx) {
  if (ctx->samp_part) return DFLASH_OK;
  const cudaError_t e = dalloc(&ctx->samp_part, static_cast<size_t>(ctx->max_rows()) * kSampleMaxSlices * kSampleWidth);
  if (e != cudaSuccess) {
    ctx->samp_part = nullptr;
    return fail(ctx, e == cudaErrorMemoryAllocation ? DFLASH_ENOMEM : DFLASH_ECUDA,
                std::string("sampling lists: ") + cudaGetErrorString(e));
  }
  return DFLASH_OK;
}

dflash_status check_sampling(dflash_ctx* ctx, float temperature, int top_k, float top_p) {
  if (!(temperature > 0.f) || !(temperature < 1e30f)) return fail(ctx, DFLASH_EINVAL, "temperature must be positive");
  if (top_k < 1 || top_k > kSampleWidth) return fail(ctx, DFLASH_EINVAL, "top_k must be in [1, 32]");
  if (!(top_p > 0.f) || top_p > 1.f) return fail(ctx, DFLASH_EINVAL, "top_p must be in (0, 1]");
  return DFLASH_OK;
}

// Target pass (dflash_target_forward): the block is the caller's ids, the
// attention causal, the block's K/V appended to the context's own pool, the
// argmax taken at every block position, the feature layers' outputs copied.
struct TargetReq {
  const int32_t* block_ids;   // device [n_seq * B]
  int pending;
  int32_t* target_ids;        // device [n_seq * B]
  uint16_t* feats;            // device [n_seq * B][n_feat * H] or null
};

dflash_status draft_impl(dflash_ctx* ctx, const int32_t* seq_ids, int n_seq, const int32_t* anchor_ids, int B,
                         int32_t* draft_ids, void* stream_v, const SampleReq* samp, const TargetReq* tgt = nullptr);

}  // namespace

dflash_status dflash_draft(dflash_ctx* ctx, const int32_t* seq_ids, int n_seq, const int32_t* anchor_ids, int B,
                           int32_t* draft_ids, void* stream_v) {
  ApiRange nvtx_range("dflash_draft");
  return draft_impl(ctx, seq_ids, n_seq, anchor_ids, B, draft_ids, stream_v, nullptr);
}

dflash_status dflash_target_forward(dflash_ctx* ctx, const int32_t* seq_ids, int n_seq, const int32_t* block_ids, int B,
                                    int pending, int32_t* target_ids, uint16_t* feats, void* stream_v) {
  ApiRange nvtx_range("dflash_target_forward");
  if (!ctx) return DFLASH_EINVAL;
  TargetReq t{block_ids, pending, target_ids, feats};
  return draft_impl(ctx, seq_ids, n_seq, nullptr, B, nullptr, stream_v, nullptr, &t);
}

dflash_status dflash_draft_sample(dflash_ctx* ctx, const int32_t* seq_ids, int n_seq, const int32_t* anchor_ids,
                                  int B, float temperature, int top_k, float top_p, const float* uniforms,
                                  int32_t* draft_ids, int32_t* q_ids, float* q_probs, void* stream_v) {
  ApiRange nvtx_range("dflash_draft_sample");
  if (!ctx) return DFLASH_EINVAL;
  dflash_status st = check_sampling(ctx, temperature, top_k, top_p);
  if (st != DFLASH_OK) return st;
  if (ctx->sel_on) return fail(ctx, DFLASH_EINVAL, "the path selector is installed (its walk is greedy)");
  if (ctx->cfg.vocab > kSampleMaxSlices * sample_slice_cols(false))
    return fail(ctx, DFLASH_EINVAL, "vocab above 524288 for sampling");
  if (B > 1 && (!uniforms || !q_ids || !q_probs)) return fail(ctx, DFLASH_EINVAL, "null uniforms or q lists");
  SampleReq r{temperature, top_p, top_k, uniforms, q_ids, q_probs};
  return draft_impl(ctx, seq_ids, n_seq, anchor_ids, B, draft_ids, stream_v, &r);
}

namespace {

dflash_status draft_impl(dflash_ctx* ctx, const int32_t* seq_ids, int n_seq, const int32_t* anchor_ids, int B,
                         int32_t* draft_ids, void* stream_v, const SampleReq* samp, const TargetReq* tgt) {
  if (!ctx) return DFLASH_EINVAL;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  const dflash_config& c = ctx->cfg;
  SeqMeta meta;
  dflash_status st = check_seqs(ctx, seq_ids, n_seq, &meta);
  if (st != DFLASH_OK) return st;
  if (B < 1 || B > c.max_block) return fail(ctx, DFLASH_EINVAL, "B out of range");
  if ((tgt != nullptr) != ctx->target)
    return fail(ctx, DFLASH_EINVAL, ctx->target ? "a target context runs dflash_target_forward"
                                                : "dflash_target_forward needs a target context");
  meta.B = B;
  if (n_seq == 0) return DFLASH_OK;
  if (tgt) {
    if (!tgt->block_ids || !tgt->target_ids) return fail(ctx, DFLASH_EINVAL, "null block_ids or target_ids");
    if (tgt->feats && (!aligned16(tgt->feats) || ctx->n_feat == 0))
      return fail(ctx, DFLASH_EINVAL, "feats not 16-byte aligned, or no feature layers");
    if (tgt->pending != 0 && tgt->pending != 1) return fail(ctx, DFLASH_EINVAL, "pending must be 0 or 1");
  } else if (!anchor_ids || (B > 1 && !draft_ids)) {
    return fail(ctx, DFLASH_EINVAL, "null anchor_ids or draft_ids");
  }
  if (samp && B > 1) {
    st = ensure_logits32(ctx);
    if (st == DFLASH_OK) st = ensure_sample_part(ctx);
    if (st != DFLASH_OK) return st;
  }
  consume_snapshot(ctx, false);
  if (tgt) {
    // the block's K/V go to positions len .. len + B - 1: reserve their pages
    // (all or nothing), as an append of B tokens does
    for (int i = 0; i < n_seq; ++i) {
      const int s = meta.slot[i];
      if (ctx->pend[s]) return fail(ctx, DFLASH_EINVAL, "target pass over a sequence with pending tokens");
      if (ctx->len_ub[s] + B > c.max_ctx) {
        consume_snapshot(ctx, true);
        if (ctx->len_ub[s] + B > c.max_ctx) return fail(ctx, DFLASH_EINVAL, "block would exceed max_ctx");
      }
      meta.row0[i] = i * B;
    }
    meta.row0[n_seq] = n_seq * B;
    auto need_pages = [&]() {
      int need = 0;
      for (int i = 0; i < n_seq; ++i) {
        const int s = meta.slot[i];
        need += std::max(0, ceil_div(ctx->len_ub[s] + B, kPage) - static_cast<int>(ctx->pages[s].size()));
      }
      return need;
    };
    if (need_pages() > static_cast<int>(ctx->free_pages.size())) {
      consume_snapshot(ctx, true);
      if (need_pages() > static_cast<int>(ctx->free_pages.size()))
        return fail(ctx, DFLASH_ENOMEM, "KV page pool exhausted");
    }
    PageUpdates& upd = *ctx->page_upd;
    upd.n = 0;
    for (int i = 0; i < n_seq; ++i) {
      const int s = meta.slot[i];
      auto& pg = ctx->pages[s];
      const int want = ceil_div(ctx->len_ub[s] + B, kPage);
      for (int k = static_cast<int>(pg.size()); k < want; ++k) {
        pg.push_back(ctx->free_pages.back());
        ctx->free_pages.pop_back();
        upd.idx[upd.n] = s * ctx->pages_per_seq + k;
        upd.page[upd.n] = pg.back();
        if (++upd.n == kPageUpdMax) {
          CK(launch_page_updates(upd, ctx->d_page_table, stream));
          upd.n = 0;
        }
      }
    }
    CK(launch_page_updates(upd, ctx->d_page_table, stream));
  }

  const int H = c.hidden, d = c.head_dim, nq = c.n_heads, nkv = c.n_kv_heads, F = c.ffn;
  const int M = n_seq * B;
  GemmWork work = gemm_work(ctx);
  const SeqState ss = seq_state(ctx);

  // attention work split from the host's length bounds
  long long tiles_ub = 0;
  for (int i = 0; i < n_seq; ++i) tiles_ub += 1LL * nkv * (ceil_div(ctx->len_ub[meta.slot[i]], kPage) + 1);
  // One wave of resident attention CTAs. Items (sequence, kv head, chunk of
  // `ch` units) are dealt largest first to the least loaded CTA, an item
  // costing its units plus kItemOverhead (query load, pipeline fill and
  // drain, partial write). The chunk size (even: the kernel consumes units in
  // pairs) is the candidate, from about one to eight chunks per CTA, whose
  // deal has the smallest makespan under the host's length bounds: equal rows
  // (batch 1) keep one chunk per CTA; rows of mixed lengths get several
  // shorter chunks, and the short row tails fill the gaps.
  int& per_sm = ctx->attn_ctas_per_sm;
  if (per_sm == 0) per_sm = attention_ctas_per_sm(d, c.kv_format == 1);
  const int grid_full = std::min(per_sm * ctx->num_sms, kSchedCtas);
  const long long item_cap = std::min<long long>(ctx->items_cap, kSchedItems);
  auto items_for = [&](int ch) {
    long long it = 0;
    for (int i = 0; i < n_seq; ++i) it += 1LL * nkv * ceil_div(ceil_div(ctx->len_ub[meta.slot[i]], kPage) + 1, ch);
    return it;
  };
  constexpr double kItemOverhead = 3.0;
  // deal chunk size ch; returns the makespan and, with `out`, the schedule
  auto deal = [&](int ch, AttnSched* out, int* grid_out) {
    std::vector<std::pair<int, uint32_t>>& items = ctx->deal_items;   // (units, record)
    items.clear();
    for (int i = 0; i < n_seq; ++i) {
      const int units = ceil_div(ctx->len_ub[meta.slot[i]], kPage) + 1;
      for (int h = 0; h < nkv; ++h)
        for (int c = 0; c * ch < units; ++c)
          items.emplace_back(std::min(ch, units - c * ch),
                             (static_cast<uint32_t>(i) << 24) | (static_cast<uint32_t>(h) << 16) | static_cast<uint32_t>(c));
    }
    std::stable_sort(items.begin(), items.end(),
                     [](const std::pair<int, uint32_t>& x, const std::pair<int, uint32_t>& y) { return x.first > y.first; });
    const int grid = static_cast<int>(std::min<long long>(static_cast<long long>(items.size()), grid_full));
    std::vector<double>& load = ctx->deal_load;
    load.assign(grid, 0.0);
    std::vector<int>& owner = ctx->deal_owner;
    owner.resize(items.size());
    using Slot = std::pair<double, int>;
    std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> heap;
    for (int c = 0; c < grid; ++c) heap.push(Slot(0.0, c));
    for (size_t k = 0; k < items.size(); ++k) {
      Slot sl = heap.top();
      heap.pop();
      owner[k] = sl.second;
      sl.first += items[k].first + kItemOverhead;
      load[sl.second] = sl.first;
      heap.push(sl);
    }
    if (out) {   // per-CTA lists in dealing order
      std::vector<int>& cnt = ctx->deal_count;
      cnt.assign(grid + 1, 0);
      for (size_t k = 0; k < items.size(); ++k) ++cnt[owner[k] + 1];
      for (int c = 0; c < grid; ++c) cnt[c + 1] += cnt[c];
      for (int c = 0; c <= grid; ++c) out->off[c] = static_cast<uint16_t>(cnt[c]);
      for (size_t k = 0; k < items.size(); ++k) out->item[cnt[owner[k]]++] = items[k].second;
      *grid_out = grid;
    }
    return *std::max_element(load.begin(), load.end());
  };
  int chunk = 0;
  double best = 0.0;
  for (int per_cta = 1; per_cta <= 8; ++per_cta) {
    int ch = std::max(2, ceil_div(tiles_ub, static_cast<long long>(per_cta) * grid_full));
    ch += ch & 1;
    if (ch == chunk || items_for(ch) > item_cap) continue;
    const double ms = deal(ch, nullptr, nullptr);
    if (chunk == 0 || ms < best) {
      chunk = ch;
      best = ms;
    }
  }
  if (chunk == 0) {   // even one chunk per CTA exceeds the partial buffers: longer chunks
    chunk = std::max(2, ceil_div(tiles_ub, grid_full));
    chunk += chunk & 1;
    while (items_for(chunk) > item_cap) chunk *= 2;
  }
  AttnSched& sched = *ctx->attn_sched;
  int attn_grid = 1;
  deal(chunk, &sched, &attn_grid);
  int max_chunks = 1;
  for (int i = 0; i < n_seq; ++i)
    max_chunks = std::max(max_chunks, ceil_div(ceil_div(ctx->len_ub[meta.slot[i]], kPage) + 1, chunk));

  const int Bb = attention_block_rows(B);
  const CUtensorMap* km = blk_map(ctx, ctx->kb, M, Bb);
  // activation descriptors: the box height is the token tile each GEMM uses
  const int sms = ctx->num_sms;
  const int n_qkv = (nq + 2 * nkv) * d, n_gu = ceil_div(F, 64) * 128;
  const CUtensorMap* hmap_qkv = act_map(ctx, ctx->hg, M, H, gemm_act_rows(M, n_qkv, H, sms));
  const CUtensorMap* hmap_gu = act_map(ctx, ctx->hg, M, H, gemm_act_rows(M, n_gu, H, sms));
  const CUtensorMap* hmap_lm = act_map(ctx, ctx->hg, M, H, gemm_act_rows(M, c.vocab, H, sms));
  const int parts = ceil_div(H, 128);
  const int rows_ld = ctx->max_rows();
  // two-tap convolutions: the O and down projections carry 2r extra rows
  // (V W of the output sites), QKV and gate/up read the convolved rows
  const bool conv = ctx->conv_on && !tgt;
  const int r2c = conv ? 2 * ctx->conv_rank : 0;
  const CUtensorMap* amap = act_map(ctx, ctx->attn, M, nq * d, gemm_act_rows(M, H + r2c, nq * d, sms));
  const CUtensorMap* fmap = act_map(ctx, ctx->act, M, F, gemm_act_rows(M, H + r2c, F, sms));
  if (!km || !hmap_qkv || !hmap_gu || !hmap_lm || !amap || !fmap)
    return fail(ctx, DFLASH_ECUDA, "activation descriptor encode failed");
  const CUtensorMap *cmap_qkv = nullptr, *cmap_gu = nullptr, *hmap_p0 = nullptr;
  if (conv) {
    cmap_qkv = act_map(ctx, ctx->conv_h, M, H, gemm_act_rows(M, n_qkv, H, sms));
    cmap_gu = act_map(ctx, ctx->conv_h, M, H, gemm_act_rows(M, n_gu, H, sms));
    hmap_p0 = act_map(ctx, ctx->hg, M, H, gemm_act_rows(M, r2c, H, sms));
    if (!cmap_qkv || !cmap_gu || !hmap_p0) return fail(ctx, DFLASH_ECUDA, "conv descriptor encode failed");
  }
  auto conv_args = [&](int l, int site) {
    ConvArgs ca;
    std::memset(&ca, 0, sizeof(ca));
    const dflash_conv_site& cs = ctx->conv_sites[4 * l + site];
    ca.M = M;
    ca.H = H;
    ca.r = ctx->conv_rank;
    ca.B = B;
    ca.base = cs.base;
    ca.U = cs.u;
    ca.inv_hidden = 1.0f / H;
    ca.eps = c.rms_eps;
    ca.status = ctx->d_status;
    return ca;
  };
  // apply kernel traffic: U (and the next V^T) slices, the rows in and out
  const double conv_w_bytes = 2.0 * H * r2c * 2;
  const size_t acc_elems = static_cast<size_t>(rows_ld) * r2c;
  // sums-of-squares parts the apply kernels write (32-column parts)
  const int conv_parts = ceil_div(H, kConvCols);
  auto conv_in_site = [&](int l, int site, const uint16_t* gain, const float* ss, int ss_parts, const float* P,
                          bool p_scaled, float* zero) -> dflash_status {
    ConvArgs ca = conv_args(l, site);
    ca.xin = ctx->x;
    ca.gin = gain;
    ca.ss = ss;
    ca.ss_parts = ss_parts;
    ca.ss_ld = rows_ld;
    ca.P = P;
    ca.p_scaled = p_scaled ? 1 : 0;
    ca.zero = zero;
    ca.out_h = ctx->conv_h;
    ProfScope ps(ctx, DFLASH_K_CONV, stream, conv_w_bytes / 2 + 6.0 * M * H + 4.0 * M * r2c,
                 2.0 * M * H * r2c + 3.0 * M * H);
    CK(launch_conv_apply(ca, stream));
    return DFLASH_OK;
  };
  auto conv_out_site = [&](int l, int site, const uint16_t* gain, float* out_ss, const uint16_t* vt,
                           float* pacc) -> dflash_status {
    ConvArgs ca = conv_args(l, site);
    ca.y = ctx->conv_yp;
    ca.ld_y = H + r2c;
    ca.x = ctx->x;
    ca.out_hg = ctx->hg;
    ca.gain = gain;
    ca.out_ss = out_ss;
    ca.out_ss_ld = rows_ld;
    ca.vt = vt;
    ca.pacc = pacc;
    ProfScope ps(ctx, DFLASH_K_CONV, stream,
                 (vt ? conv_w_bytes : conv_w_bytes / 2) + 1.0 * M * (H + r2c) * 4 + 10.0 * M * H +
                     (vt ? 4.0 * M * r2c : 0),
                 2.0 * M * H * r2c * (vt ? 1.5 : 1.0) + 6.0 * M * H);
    CK(launch_conv_apply(ca, stream));
    return DFLASH_OK;
  };
  auto vt_of = [&](int l, int which) {   // which 0: V_ai^T, 1: V_fi^T
    return ctx->conv_vt + static_cast<size_t>(2 * l + which) * H * r2c;
  };
  AttnMaps attn_maps;
  attn_maps.pool_k = ctx->m_pool;
  attn_maps.pool_vt = ctx->m_pool_vt;
  attn_maps.kblk = *km;
  attn_maps.vblk = ctx->m_vblk;

  double ctx_tokens = 0, attn_flops = 0;
  for (int i = 0; i < n_seq; ++i) {
    ctx_tokens += ctx->len_ub[meta.slot[i]];
    attn_flops += 4.0 * B * nq * d * (ctx->len_ub[meta.slot[i]] + B);
  }
  // context K/V per token and kv head: 4 d bytes (bf16) or 2 d codes + 2 d/32 fp16 scales (8-bit pages)
  const double kv_token_head = c.kv_format == 1 ? 2.125 * d : 4.0 * d;
  const double attn_bytes = ctx_tokens * nkv * kv_token_head + 1.0 * M * nkv * d * 4 + 1.0 * M * nq * d * 2;
  {
    ProfScope ps(ctx, DFLASH_K_NORM, stream, 8.0 * M * H, 0);
    CK(launch_embed(ctx->w.embed, anchor_ids, c.mask_id, tgt ? tgt->block_ids : nullptr, c.vocab, meta, H,
                    ctx->layers[0].g_attn, ctx->x, ctx->hg, ctx->ssA, ctx->d_status, stream));
  }
  for (int l = 0; l < c.n_layers; ++l) {
    const dflash_layer_weights& L = ctx->layers[l];
    if (conv) {   // h = Conv_ai(RMSNorm(x)); layer 0's products V_ai x from one GEMM over the embedding rows
      if (l == 0) {
        AMaps am;
        am.m[0] = ctx->m_vai0;
        GemmEpi e = base_epi(ctx, EPI_F32_STORE);
        e.out_f32 = ctx->conv_p;
        e.ld_out = r2c;
        e.in_ss = ctx->ssA;
        e.in_ss_parts = 1;
        e.in_ss_ld = rows_ld;
        ProfScope ps(ctx, DFLASH_K_CONV, stream, gemm_bytes(M, r2c, H, r2c, 4), 2.0 * M * r2c * H);
        CK(launch_gemm(am, stacked({r2c}), *hmap_p0, M, r2c, H, 0, e, work, ctx->num_sms, stream));
      }
      // P: layer 0's from the GEMM (scaled); later layers' accumulated by the
      // previous layer's feed-forward output site (accumulator 1). Clears
      // accumulator 0 for this layer's attention output site.
      const dflash_status st = conv_in_site(l, 0, L.g_attn, ctx->ssA, l == 0 ? 1 : conv_parts,
                                            l == 0 ? ctx->conv_p : ctx->conv_acc + acc_elems, l == 0, ctx->conv_acc);
      if (st != DFLASH_OK) return st;
    }
    {  // q, k, v with RoPE at positions len .. len+B-1
      AMaps am;
      am.m[0] = ctx->m_wq[l];
      am.m[1] = ctx->m_wk[l];
      am.m[2] = ctx->m_wv[l];
      ARegions rg = stacked({nq * d, nkv * d, nkv * d});
      rg.pair = d / 2;
      GemmEpi e = base_epi(ctx, EPI_QKV_ROPE);
      e.qkv_f16 = c.kv_format == 1;   // the 8-bit pages' attention runs in fp16
      e.out_q = ctx->q;
      e.out_k = ctx->kb;
      e.out_v = ctx->vb;
      e.meta = meta;
      e.in_ss = conv ? nullptr : ctx->ssA;   // the convolved rows are normalised already
      e.in_ss_parts = l == 0 ? 1 : parts;
      e.in_ss_ld = rows_ld;
      const double nw = 1.0 * (nq + 2 * nkv) * d;
      ProfScope ps(ctx, DFLASH_K_QKV, stream, gemm_bytes(M, nw, H, nw, 2), 2.0 * M * nw * H);
      CK(launch_gemm(am, rg, conv ? *cmap_qkv : *hmap_qkv, M, n_qkv, H, 0, e, work, ctx->num_sms, stream));
    }
    if (tgt) {   // the block's K/V into the target's own cache
      ProfScope ps(ctx, DFLASH_K_OTHER, stream, 4.0 * M * nkv * d * 2, 0);
      CK(launch_block_kv_append(meta, ss, l, ctx->kb, ctx->vb, ctx->pool, c.max_pages, nkv, d, ctx->d_status, stream));
    }
    {  // non-causal attention over the injected context and the block
      AttnArgs a;
      std::memset(&a, 0, sizeof(a));
      a.meta = meta;
      a.seqs = ss;
      a.layer = l;
      a.n_q_heads = nq;
      a.n_kv_heads = nkv;
      a.head_dim = d;
      a.pool_pages = c.max_pages;
      a.chunk_tiles = chunk;
      a.max_chunks = max_chunks;
      a.items_cap = ctx->items_cap;
      a.rows_pad = 16 * ceil_div((nq / nkv) * B, 16);
      a.spread = (nq / nkv) * B <= 64;
      a.causal = tgt ? 1 : 0;
      a.q8 = c.kv_format == 1;
      a.q = ctx->q;
      a.pool = ctx->pool;
      a.part_o = ctx->part_o;
      a.part_ml = ctx->part_ml;
      a.out = ctx->attn;
      a.status = ctx->d_status;
      {
        ProfScope ps(ctx, DFLASH_K_ATTN, stream, attn_bytes, attn_flops);
        CK(launch_attention(attn_maps, a, sched, attn_grid, 0, stream));
      }
      {
        ProfScope ps(ctx, DFLASH_K_ATTN_COMBINE, stream, 2.0 * M * nq * d, 0);
        CK(launch_attention(attn_maps, a, sched, attn_grid, 1, stream));
      }
    }
    if (conv) {   // [attn W_o^T | attn (V_ao W_o)^T], then x += Conv_ao, then h = Conv_fi(RMSNorm(x))
      AMaps am;
      am.m[0] = ctx->m_wo[l];
      am.m[1] = ctx->m_fold_o[l];
      GemmEpi e = base_epi(ctx, EPI_F32_STORE);
      e.out_f32 = ctx->conv_yp;
      e.ld_out = H + r2c;
      {
        ProfScope ps(ctx, DFLASH_K_O, stream, gemm_bytes(M, H + r2c, nq * d, H + r2c, 4), 2.0 * M * (H + r2c) * nq * d);
        CK(launch_gemm(am, stacked({H, r2c}), *amap, M, H + r2c, nq * d, 0, e, work, ctx->num_sms, stream));
      }
      dflash_status st = conv_out_site(l, 1, L.g_ffn, ctx->ssB, vt_of(l, 1), ctx->conv_acc);
      if (st == DFLASH_OK)
        st = conv_in_site(l, 2, L.g_ffn, ctx->ssB, conv_parts, ctx->conv_acc, false, ctx->conv_acc + acc_elems);
      if (st != DFLASH_OK) return st;
    } else {  // x += attn W_o^T; the FFN's RMSNorm input is folded into the epilogue
      AMaps am;
      am.m[0] = ctx->m_wo[l];
      GemmEpi e = base_epi(ctx, EPI_RESID);
      e.out_f32 = ctx->x;
      e.ld_out = H;
      e.out_hg = ctx->hg;
      e.gain = L.g_ffn;
      e.out_ss = ctx->ssB;
      e.out_ss_ld = rows_ld;
      ProfScope ps(ctx, DFLASH_K_O, stream, gemm_bytes(M, H, nq * d, H, 10), 2.0 * M * H * nq * d);
      CK(launch_gemm(am, stacked({H}), *amap, M, H, nq * d, 0, e, work, ctx->num_sms, stream));
    }
    {  // act = SiLU(h W_gate^T) * (h W_up^T)
      AMaps am;
      am.m[0] = ctx->m_wg[l];
      am.m[1] = ctx->m_wu[l];
      ARegions rg;
      std::memset(&rg, 0, sizeof(rg));
      rg.n_regions = 2;
      rg.paired = 1;
      rg.pair = 64;
      GemmEpi e = base_epi(ctx, EPI_SWIGLU);
      e.out_act = ctx->act;
      e.n_valid = F;
      e.in_ss = conv ? nullptr : ctx->ssB;
      e.in_ss_parts = parts;
      e.in_ss_ld = rows_ld;
      ProfScope ps(ctx, DFLASH_K_GATEUP, stream, gemm_bytes(M, 2.0 * F, H, F, 2), 4.0 * M * F * H);
      CK(launch_gemm(am, rg, conv ? *cmap_gu : *hmap_gu, M, n_gu, H, 0, e, work, ctx->num_sms, stream));
    }
    if (conv) {   // [act W_down^T | act (V_fo W_down)^T], then x += Conv_fo (+ the next layer's V_ai products)
      AMaps am;
      am.m[0] = ctx->m_wd[l];
      am.m[1] = ctx->m_fold_d[l];
      GemmEpi e = base_epi(ctx, EPI_F32_STORE);
      e.out_f32 = ctx->conv_yp;
      e.ld_out = H + r2c;
      {
        ProfScope ps(ctx, DFLASH_K_DOWN, stream, gemm_bytes(M, H + r2c, F, H + r2c, 4), 2.0 * M * (H + r2c) * F);
        CK(launch_gemm(am, stacked({H, r2c}), *fmap, M, H + r2c, F, 0, e, work, ctx->num_sms, stream));
      }
      const bool last = l + 1 == c.n_layers;
      const dflash_status st = conv_out_site(l, 3, last ? ctx->w.g_final : ctx->layers[l + 1].g_attn, ctx->ssA,
                                             last ? nullptr : vt_of(l + 1, 0), ctx->conv_acc + acc_elems);
      if (st != DFLASH_OK) return st;
    } else {  // x += act W_down^T; the next RMSNorm (next layer's input, or the final norm) is folded in
      AMaps am;
      am.m[0] = ctx->m_wd[l];
      GemmEpi e = base_epi(ctx, EPI_RESID);
      e.out_f32 = ctx->x;
      e.ld_out = H;
      e.out_hg = ctx->hg;
      e.gain = l + 1 < c.n_layers ? ctx->layers[l + 1].g_attn : ctx->w.g_final;
      e.out_ss = ctx->ssA;
      e.out_ss_ld = rows_ld;
      ProfScope ps(ctx, DFLASH_K_DOWN, stream, gemm_bytes(M, H, F, H, 10), 2.0 * M * H * F);
      CK(launch_gemm(am, stacked({H}), *fmap, M, H, F, 0, e, work, ctx->num_sms, stream));
    }
    if (tgt && tgt->feats && ctx->feat_slot[l] >= 0) {   // this layer's output is a feature
      ProfScope ps(ctx, DFLASH_K_OTHER, stream, 6.0 * M * H, 0);
      CK(launch_feat_copy(ctx->x, M, H, tgt->feats, ctx->n_feat * H, ctx->feat_slot[l] * H, stream));
    }
  }
  ctx->last_rows = M;
  ctx->last_draft_rows = tgt ? M : n_seq * (B - 1);
  ctx->last_sel_rows = ctx->sel_on && !samp && !tgt ? n_seq * (B - 1) : 0;
  if (tgt) {
    // LM head with the argmax at every block position (final norm folded in)
    AMaps am;
    am.m[0] = ctx->m_lm;
    GemmEpi e = base_epi(ctx, EPI_ARGMAX);
    e.keys = ctx->keys;
    e.done = ctx->done;
    e.out_ids = tgt->target_ids;
    e.out_logit = ctx->top_logit;
    e.argmax_skip_B = 0;
    e.in_ss = ctx->ssA;
    e.in_ss_parts = conv ? conv_parts : parts;
    e.in_ss_ld = rows_ld;
    {
      ProfScope ps(ctx, DFLASH_K_LMHEAD, stream, gemm_bytes(M, c.vocab, H, 1, 8), 2.0 * M * c.vocab * H);
      CK(launch_gemm(am, stacked({c.vocab}), *hmap_lm, M, c.vocab, H, 0, e, work, ctx->num_sms, stream));
    }
    // the block's tokens become pending (verify commits tau) or committed
    {
      ProfScope ps(ctx, DFLASH_K_OTHER, stream, 8.0 * n_seq, 0);
      CK(launch_fuse_advance(meta, ss, tgt->pending, stream));
    }
    for (int i = 0; i < n_seq; ++i) {
      const int s = meta.slot[i];
      if (tgt->pending) ctx->pend[s] += B;
      else {
        ctx->len_ub[s] += B;
        ctx->added_since[s] += B;
      }
    }
  } else if (B > 1 && samp) {
    // LM head into fp32 rows (final RMSNorm scale applied), then the 32
    // largest logits of every masked row, the filter and the draw
    const int Md = n_seq * (B - 1);
    const CUtensorMap* hmap_s = act_map(ctx, ctx->hg, M, H, gemm_act_rows(M, c.vocab, H, sms));
    if (!hmap_s) return fail(ctx, DFLASH_ECUDA, "activation descriptor encode failed");
    AMaps am;
    am.m[0] = ctx->m_lm;
    GemmEpi e = base_epi(ctx, EPI_F32_STORE);
    e.out_f32 = ctx->sel_logits;
    e.ld_out = ctx->sel_ld;
    e.in_ss = ctx->ssA;
    e.in_ss_parts = conv ? conv_parts : parts;
    e.in_ss_ld = rows_ld;
    {
      ProfScope ps(ctx, DFLASH_K_LMHEAD, stream, gemm_bytes(M, c.vocab, H, c.vocab, 4), 2.0 * M * c.vocab * H);
      CK(launch_gemm(am, stacked({c.vocab}), *hmap_s, M, c.vocab, H, 0, e, work, ctx->num_sms, stream));
    }
    FilterArgs fa;
    fa.slices = ceil_div(c.vocab, sample_slice_cols(false));
    fa.part = ctx->samp_part;
    fa.inv_temperature = 1.f / samp->temperature;
    fa.top_k = samp->top_k;
    fa.top_p = samp->top_p;
    fa.uniforms = samp->uniforms;
    fa.out_ids = samp->q_ids;
    fa.out_probs = samp->q_probs;
    fa.drawn = draft_ids;
    ProfScope ps(ctx, DFLASH_K_SAMPLE, stream, 4.0 * Md * c.vocab + 8.0 * Md * fa.slices * kSampleWidth * 2 +
                 8.0 * Md * kSampleWidth + 8.0 * Md, 0, 2);
    CK(launch_sample_filter(ctx->sel_logits, false, ctx->sel_ld, c.vocab, Md, B, ctx->samp_part, fa, stream));
  } else if (B > 1 && ctx->sel_on) {
    // LM head and the selector's context gate H = W_H h~ in one GEMM over all
    // block rows, final RMSNorm scale applied: logits in columns [0, V), H in
    // [sel_hcol, sel_hcol + 256). Then top-16, pair scores and the walk.
    const int Md = n_seq * (B - 1);
    const int n_out = ctx->sel_hcol + kSelDim;
    const CUtensorMap* hmap_sel = act_map(ctx, ctx->hg, M, H, gemm_act_rows(M, n_out, H, sms));
    if (!hmap_sel) return fail(ctx, DFLASH_ECUDA, "activation descriptor encode failed");
    AMaps am;
    am.m[0] = ctx->m_lm;
    am.m[1] = ctx->m_wh;
    GemmEpi e = base_epi(ctx, EPI_F32_STORE);
    e.out_f32 = ctx->sel_logits;
    e.ld_out = ctx->sel_ld;
    e.in_ss = ctx->ssA;
    e.in_ss_parts = conv ? conv_parts : parts;
    e.in_ss_ld = rows_ld;
    {
      ProfScope ps(ctx, DFLASH_K_LMHEAD, stream, gemm_bytes(M, n_out, H, n_out, 4), 2.0 * M * n_out * H);
      CK(launch_gemm(am, stacked({c.vocab, kSelDim}), *hmap_sel, M, n_out, H, 0, e, work, ctx->num_sms, stream));
    }
    SelectArgs sa;
    sa.n_seq = n_seq;
    sa.B = B;
    sa.V = c.vocab;
    sa.logits = ctx->sel_logits;
    sa.ld = ctx->sel_ld;
    sa.h_col = ctx->sel_hcol;
    sa.slices = ceil_div(c.vocab, kSelSliceCols);
    sa.part = ctx->sel_part;
    sa.table = ctx->sel_table;
    sa.anchors = anchor_ids;
    sa.scores = ctx->sel_scores;
    sa.cand = ctx->sel_cand;
    sa.cand_u = ctx->sel_cand_u;
    sa.next = ctx->sel_next;
    sa.top_logit = ctx->top_logit;
    sa.tickets = ctx->sel_tickets;
    sa.draft_ids = draft_ids;
    sa.status = ctx->d_status;
    // logits read once, the 16-key lists, candidate rows of the A|B table,
    // H rows, the scores and ids
    const double sel_bytes = 4.0 * Md * (c.vocab + kSelDim) + 2.0 * 8 * Md * sa.slices * kSelK +
                             4.0 * Md * kSelK * 2 * kSelDim + 4.0 * Md * kSelK * kSelK + 4.0 * Md;
    ProfScope ps(ctx, DFLASH_K_SELECT, stream, sel_bytes, 2.0 * Md * kSelK * kSelK * kSelDim, 2);
    CK(launch_path_select(sa, stream));
  } else if (B > 1) {
    // LM head over all block rows (the anchor rows are skipped in the epilogue),
    // final RMSNorm folded in: the argmax is taken on the unscaled logits (a
    // positive per-row scale does not move it) and the winning logit is scaled.
    const int Md = n_seq * (B - 1);
    AMaps am;
    am.m[0] = ctx->m_lm;
    GemmEpi e = base_epi(ctx, EPI_ARGMAX);
    e.keys = ctx->keys;
    e.done = ctx->done;
    e.out_ids = draft_ids;
    e.out_logit = ctx->top_logit;
    e.argmax_skip_B = B;
    e.in_ss = ctx->ssA;
    e.in_ss_parts = conv ? conv_parts : parts;
    e.in_ss_ld = rows_ld;
    ProfScope ps(ctx, DFLASH_K_LMHEAD, stream, gemm_bytes(Md, c.vocab, H, 1, 8), 2.0 * Md * c.vocab * H);
    CK(launch_gemm(am, stacked({c.vocab}), *hmap_lm, M, c.vocab, H, 0, e, work, ctx->num_sms, stream));
  }
  return DFLASH_OK;
}

// After a verify launch: the host's length bounds take every pending token
// (the device commits tau of them), and a snapshot of the exact lengths is
// requested to tighten the bounds later.
dflash_status commit_host_side(dflash_ctx* ctx, const SeqMeta& meta, int n_seq, cudaStream_t stream) {
  bool had_pending = false;
  for (int i = 0; i < n_seq; ++i) {
    const int s = meta.slot[i];
    had_pending |= ctx->pend[s] > 0;
    ctx->len_ub[s] += ctx->pend[s];
    ctx->pend[s] = 0;
  }
  if (had_pending) {
    consume_snapshot(ctx, false);
    if (!ctx->snap_pending) {
      CK(cudaMemcpyAsync(ctx->h_snap, ctx->d_len, ctx->cfg.max_seqs * sizeof(int), cudaMemcpyDeviceToHost, stream));
      CK(cudaEventRecord(ctx->snap_event, stream));
      std::fill(ctx->added_since.begin(), ctx->added_since.end(), 0);
      ctx->snap_pending = true;
    }
  }
  return DFLASH_OK;
}

}  // namespace

dflash_status dflash_verify(dflash_ctx* ctx, const int32_t* seq_ids, int n_seq, int B, const int32_t* draft_ids,
                            const int32_t* target_ids, int32_t* tau, int32_t* bonus, void* stream_v) {
  ApiRange nvtx_range("dflash_verify");
  if (!ctx) return DFLASH_EINVAL;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  SeqMeta meta;
  dflash_status st = check_seqs(ctx, seq_ids, n_seq, &meta);
  if (st != DFLASH_OK) return st;
  if (B < 1 || B > ctx->cfg.max_block) return fail(ctx, DFLASH_EINVAL, "B out of range");
  meta.B = B;
  if (n_seq == 0) return DFLASH_OK;
  if ((B > 1 && !draft_ids) || !target_ids || !tau || !bonus) return fail(ctx, DFLASH_EINVAL, "null pointer");
  {
    ProfScope ps(ctx, DFLASH_K_VERIFY, stream, 4.0 * n_seq * (2 * B + 2), 0);
    CK(launch_verify(meta, seq_state(ctx), draft_ids, target_ids, tau, bonus, stream));
  }
  return commit_host_side(ctx, meta, n_seq, stream);
}

dflash_status dflash_rows_argmax_bf16(const uint16_t* logits, int rows, int cols, int32_t* out, void* stream) {
  ApiRange nvtx_range("dflash_rows_argmax_bf16");
  if (rows < 0 || cols < 1) return DFLASH_EINVAL;
  if (rows > 0 && (!logits || !out)) return DFLASH_EINVAL;
  return launch_rows_argmax_bf16(logits, rows, cols, out, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? DFLASH_OK
             : DFLASH_ECUDA;
}

dflash_status dflash_debug_read_kv(dflash_ctx* ctx, int layer, int seq, int pos0, int n, uint16_t* k_out,
                                   uint16_t* v_out) {
  if (!ctx) return DFLASH_EINVAL;
  const dflash_config& c = ctx->cfg;
  if (layer < 0 || layer >= c.n_layers || seq < 0 || seq >= c.max_seqs || pos0 < 0 || n < 0)
    return fail(ctx, DFLASH_EINVAL, "argument out of range");
  CK(cudaDeviceSynchronize());
  int len = 0, pend = 0;
  CK(cudaMemcpy(&len, ctx->d_len + seq, sizeof(int), cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(&pend, ctx->d_pend + seq, sizeof(int), cudaMemcpyDeviceToHost));
  if (pos0 + n > len + pend) return fail(ctx, DFLASH_EINVAL, "positions beyond the cached tokens");
  const int d = c.head_dim, nkv = c.n_kv_heads;
  if (c.kv_format == 1) {   // decoded 8-bit blocks, rounded to bf16
    std::vector<int8_t> kc(static_cast<size_t>(n) * nkv * d), vc(kc.size());
    std::vector<uint16_t> ks(static_cast<size_t>(n) * nkv * (d / 32)), vs(ks.size());
    dflash_status st = dflash_debug_read_kv_q8(ctx, layer, seq, pos0, n, kc.data(), ks.data(), vc.data(), vs.data());
    if (st != DFLASH_OK) return st;
    auto h2f = [](uint16_t h) {   // fp16 -> fp32
      const uint32_t sgn = (h & 0x8000u) << 16, ex = (h >> 10) & 0x1Fu, mant = h & 0x3FFu;
      float v;
      if (ex == 0) v = std::ldexp(static_cast<float>(mant), -24);
      else if (ex == 31) v = mant ? NAN : INFINITY;
      else v = std::ldexp(static_cast<float>(mant | 0x400u), static_cast<int>(ex) - 25);
      return sgn ? -v : v;
    };
    auto f2bf = [](float f) {   // round to nearest even
      uint32_t u;
      std::memcpy(&u, &f, 4);
      u += 0x7FFFu + ((u >> 16) & 1u);
      return static_cast<uint16_t>(u >> 16);
    };
    for (size_t e = 0; e < kc.size(); ++e) {
      const size_t blk = e / 32;
      if (k_out) k_out[e] = f2bf(static_cast<float>(kc[e]) * h2f(ks[blk]));
      if (v_out) v_out[e] = f2bf(static_cast<float>(vc[e]) * h2f(vs[blk]));
    }
    return DFLASH_OK;
  }
  const size_t page_elems = static_cast<size_t>(2) * nkv * kPage * d;
  std::vector<uint16_t> buf(page_elems);
  int cur_page = -1;
  for (int t = 0; t < n; ++t) {
    const int pos = pos0 + t;
    const int pi = pos / kPage;
    if (pi >= static_cast<int>(ctx->pages[seq].size())) return fail(ctx, DFLASH_EINVAL, "position not paged");
    const int page = ctx->pages[seq][pi];
    if (page != cur_page) {
      const size_t off = (static_cast<size_t>(layer) * c.max_pages + page) * page_elems;
      CK(cudaMemcpy(buf.data(), ctx->pool + off, page_elems * 2, cudaMemcpyDeviceToHost));
      cur_page = page;
    }
    const int slot = pos % kPage;
    for (int h = 0; h < nkv; ++h) {
      // keys [n_kv][64 slots][d], then values transposed [n_kv][d][64 slots]
      const uint16_t* ks = buf.data() + (static_cast<size_t>(h) * kPage + slot) * d;
      const uint16_t* vs = buf.data() + static_cast<size_t>(nkv) * kPage * d + static_cast<size_t>(h) * d * kPage + slot;
      if (k_out) std::memcpy(k_out + (static_cast<size_t>(t) * nkv + h) * d, ks, d * 2);
      if (v_out)
        for (int di = 0; di < d; ++di) v_out[(static_cast<size_t>(t) * nkv + h) * d + di] = vs[static_cast<size_t>(di) * kPage];
    }
  }
  return DFLASH_OK;
}

dflash_status dflash_debug_read_kv_q8(dflash_ctx* ctx, int layer, int seq, int pos0, int n, int8_t* k_codes,
                                      uint16_t* k_scales, int8_t* v_codes, uint16_t* v_scales) {
  if (!ctx) return DFLASH_EINVAL;
  const dflash_config& c = ctx->cfg;
  if (c.kv_format != 1) return fail(ctx, DFLASH_EINVAL, "the cache is not in the 8-bit format");
  if (layer < 0 || layer >= c.n_layers || seq < 0 || seq >= c.max_seqs || pos0 < 0 || n < 0)
    return fail(ctx, DFLASH_EINVAL, "argument out of range");
  CK(cudaDeviceSynchronize());
  int len = 0, pend = 0;
  CK(cudaMemcpy(&len, ctx->d_len + seq, sizeof(int), cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(&pend, ctx->d_pend + seq, sizeof(int), cudaMemcpyDeviceToHost));
  if (pos0 + n > len + pend) return fail(ctx, DFLASH_EINVAL, "positions beyond the cached tokens");
  const int d = c.head_dim, nkv = c.n_kv_heads, nb = d / 32;
  const size_t hb = q8_head_bytes(d);
  std::vector<uint8_t> buf(hb * nkv);
  const uint8_t* pool = reinterpret_cast<const uint8_t*>(ctx->pool);
  int cur_page = -1;
  for (int t = 0; t < n; ++t) {
    const int pos = pos0 + t;
    const int pi = pos / kPage;
    if (pi >= static_cast<int>(ctx->pages[seq].size())) return fail(ctx, DFLASH_EINVAL, "position not paged");
    const int page = ctx->pages[seq][pi];
    if (page != cur_page) {
      CK(cudaMemcpy(buf.data(), pool + (static_cast<size_t>(layer) * c.max_pages + page) * nkv * hb, hb * nkv,
                    cudaMemcpyDeviceToHost));
      cur_page = page;
    }
    const int slot = pos % kPage;
    for (int h = 0; h < nkv; ++h) {
      const uint8_t* r = buf.data() + h * hb;
      const uint16_t* ksc = reinterpret_cast<const uint16_t*>(r + q8_kscale_off(d));
      const uint16_t* vsc = reinterpret_cast<const uint16_t*>(r + q8_vscale_off(d));
      for (int di = 0; di < d; ++di) {
        const size_t o = (static_cast<size_t>(t) * nkv + h) * d + di;
        // stored offset-binary (code + 128)
        if (k_codes) k_codes[o] = static_cast<int8_t>(static_cast<int>(r[slot * d + di]) - 128);
        if (v_codes)
          v_codes[o] = static_cast<int8_t>(static_cast<int>(r[q8_vcode_off(d) + static_cast<size_t>(di) * kPage + slot]) - 128);
      }
      for (int b = 0; b < nb; ++b) {
        const size_t o = (static_cast<size_t>(t) * nkv + h) * nb + b;
        if (k_scales) k_scales[o] = ksc[slot * nb + b];
        if (v_scales) v_scales[o] = vsc[b * kPage + slot];
      }
    }
  }
  return DFLASH_OK;
}

dflash_status dflash_sample_filter(dflash_ctx* ctx, const uint16_t* logits, int rows, int cols, float temperature,
                                   int top_k, float top_p, const float* uniforms, int32_t* out_ids, float* out_probs,
                                   int32_t* drawn, void* stream_v) {
  ApiRange nvtx_range("dflash_sample_filter");
  if (!ctx) return DFLASH_EINVAL;
  dflash_status st = check_sampling(ctx, temperature, top_k, top_p);
  if (st != DFLASH_OK) return st;
  if (rows < 0 || rows > ctx->max_rows()) return fail(ctx, DFLASH_EINVAL, "rows outside [0, max_batch * max_block]");
  if (rows == 0) return DFLASH_OK;
  if (cols < kSampleWidth || cols % 8 || cols > kSampleMaxSlices * sample_slice_cols(true))
    return fail(ctx, DFLASH_EINVAL, "cols must be a multiple of 8 in [32, 524288]");
  if (!logits || !out_ids || !out_probs || (drawn && !uniforms)) return fail(ctx, DFLASH_EINVAL, "null pointer");
  if (!aligned16(logits)) return fail(ctx, DFLASH_EINVAL, "logits not 16-byte aligned");
  st = ensure_sample_part(ctx);
  if (st != DFLASH_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  FilterArgs fa;
  fa.slices = ceil_div(cols, sample_slice_cols(true));
  fa.part = ctx->samp_part;
  fa.inv_temperature = 1.f / temperature;
  fa.top_k = top_k;
  fa.top_p = top_p;
  fa.uniforms = uniforms;
  fa.out_ids = out_ids;
  fa.out_probs = out_probs;
  fa.drawn = drawn;
  ProfScope ps(ctx, DFLASH_K_SAMPLE, stream, 2.0 * rows * cols + 16.0 * rows * fa.slices * kSampleWidth +
               8.0 * rows * kSampleWidth, 0, 2);
  CK(launch_sample_filter(logits, true, cols, cols, rows, 0, ctx->samp_part, fa, stream));
  return DFLASH_OK;
}

dflash_status dflash_verify_sample(dflash_ctx* ctx, const int32_t* seq_ids, int n_seq, int B, const int32_t* draft_ids,
                                   const int32_t* q_ids, const float* q_probs, const int32_t* p_ids,
                                   const float* p_probs, const float* u_accept, const float* u_resample,
                                   int32_t* tau, int32_t* bonus, void* stream_v) {
  ApiRange nvtx_range("dflash_verify_sample");
  if (!ctx) return DFLASH_EINVAL;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  SeqMeta meta;
  dflash_status st = check_seqs(ctx, seq_ids, n_seq, &meta);
  if (st != DFLASH_OK) return st;
  if (B < 1 || B > ctx->cfg.max_block) return fail(ctx, DFLASH_EINVAL, "B out of range");
  meta.B = B;
  if (n_seq == 0) return DFLASH_OK;
  if ((B > 1 && (!draft_ids || !q_ids || !q_probs || !u_accept)) || !p_ids || !p_probs || !u_resample || !tau ||
      !bonus)
    return fail(ctx, DFLASH_EINVAL, "null pointer");
  VerifySampleArgs a;
  a.drafts = draft_ids;
  a.q_ids = q_ids;
  a.q_probs = q_probs;
  a.p_ids = p_ids;
  a.p_probs = p_probs;
  a.u_accept = u_accept;
  a.u_resample = u_resample;
  a.tau = tau;
  a.bonus = bonus;
  a.status = ctx->d_status;
  {
    ProfScope ps(ctx, DFLASH_K_VERIFY, stream, 4.0 * n_seq * (2 * B + 2) + 8.0 * n_seq * (2 * B - 1) * kSampleWidth,
                 0);
    CK(launch_verify_sample(meta, seq_state(ctx), a, stream));
  }
  return commit_host_side(ctx, meta, n_seq, stream);
}

dflash_status dflash_set_path_selector(dflash_ctx* ctx, const uint16_t* w_a, const uint16_t* w_b,
                                       const uint16_t* w_h, int dim, void* stream_v) {
  ApiRange nvtx_range("dflash_set_path_selector");
  if (!ctx) return DFLASH_EINVAL;
  if (ctx->target) return fail(ctx, DFLASH_EINVAL, "the path selector belongs to a drafter context");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  const dflash_config& c = ctx->cfg;
  const int H = c.hidden;
  if (!w_a && !w_b && !w_h) {
    ctx->sel_on = false;
    return DFLASH_OK;
  }
  if (!w_a || !w_b || !w_h) return fail(ctx, DFLASH_EINVAL, "w_a, w_b, w_h must be all set or all NULL");
  if (dim != kSelDim) return fail(ctx, DFLASH_EINVAL, "selector width must be 256");
  if (c.vocab < kSelK || c.vocab > kSelMaxSlices * kSelSliceCols)
    return fail(ctx, DFLASH_EINVAL, "vocab outside [16, 524288] for the path selector");
  if (!aligned16(w_a) || !aligned16(w_b) || !aligned16(w_h)) return fail(ctx, DFLASH_EINVAL, "weights not 16-byte aligned");
  const size_t rows = ctx->max_rows();
  dflash_status lst = ensure_logits32(ctx);
  if (lst != DFLASH_OK) return lst;
  if (!ctx->sel_table) {
    cudaError_t e = dalloc(&ctx->sel_table, static_cast<size_t>(c.vocab) * 2 * kSelDim);
    if (e == cudaSuccess) e = dalloc(&ctx->sel_part, rows * kSelMaxSlices * kSelK);
    if (e == cudaSuccess) e = dalloc(&ctx->sel_scores, rows * kSelK * kSelK);
    if (e == cudaSuccess) e = dalloc(&ctx->sel_cand, rows * kSelK);
    if (e == cudaSuccess) e = dalloc(&ctx->sel_cand_u, rows * kSelK);
    if (e == cudaSuccess) e = dalloc(&ctx->sel_next, rows * kSelK);
    if (e == cudaSuccess) e = dalloc(&ctx->sel_tickets, c.max_batch);
    if (e == cudaSuccess) e = cudaMemset(ctx->sel_tickets, 0, c.max_batch * sizeof(int));
    if (e != cudaSuccess) {
      void* ps[] = {ctx->sel_table, ctx->sel_part, ctx->sel_scores, ctx->sel_cand, ctx->sel_cand_u,
                    ctx->sel_tickets, ctx->sel_next};
      for (void* p : ps)
        if (p) cudaFree(p);
      ctx->sel_table = nullptr;
      ctx->sel_part = nullptr;
      ctx->sel_scores = nullptr;
      ctx->sel_cand = nullptr;
      ctx->sel_cand_u = nullptr;
      ctx->sel_tickets = nullptr;
      ctx->sel_next = nullptr;
      return fail(ctx, e == cudaErrorMemoryAllocation ? DFLASH_ENOMEM : DFLASH_ECUDA,
                  std::string("selector buffers: ") + cudaGetErrorString(e));
    }
  }
  ctx->sel_on = false;
  CUtensorMap m_wa, m_wb;
  if (!encode_2d(&m_wa, w_a, kSelDim, H, kWeightBoxRows) || !encode_2d(&m_wb, w_b, kSelDim, H, kWeightBoxRows) ||
      !encode_2d(&ctx->m_wh, w_h, kSelDim, H, kWeightBoxRows))
    return fail(ctx, DFLASH_ECUDA, "selector weight descriptor encode failed");
  // table[v] = (W_A E[v] | W_B E[v]): the embedding rows are the tokens of a
  // GEMM against the stacked [W_A; W_B], in chunks of at most 1024 rows
  constexpr int kChunk = 1024;
  GemmWork work = gemm_work(ctx);
  AMaps am;
  am.m[0] = m_wa;
  am.m[1] = m_wb;
  for (int r0 = 0; r0 < c.vocab; r0 += kChunk) {
    const int M = std::min(kChunk, c.vocab - r0);
    CUtensorMap xm;
    if (!encode_2d(&xm, ctx->w.embed + static_cast<size_t>(r0) * H, M, H,
                   gemm_act_rows(M, 2 * kSelDim, H, ctx->num_sms)))
      return fail(ctx, DFLASH_ECUDA, "embedding descriptor encode failed");
    GemmEpi e = base_epi(ctx, EPI_F32_STORE);
    e.out_f32 = ctx->sel_table + static_cast<size_t>(r0) * 2 * kSelDim;
    e.ld_out = 2 * kSelDim;
    CK(launch_gemm(am, stacked({kSelDim, kSelDim}), xm, M, 2 * kSelDim, H, 0, e, work, ctx->num_sms, stream));
  }
  CK(cudaStreamSynchronize(stream));
  ctx->sel_on = true;
  return DFLASH_OK;
}

dflash_status dflash_set_conv(dflash_ctx* ctx, const dflash_conv_site* sites, int rank, void* stream_v) {
  ApiRange nvtx_range("dflash_set_conv");
  if (!ctx) return DFLASH_EINVAL;
  if (ctx->target) return fail(ctx, DFLASH_EINVAL, "the two-tap convolutions belong to a drafter context");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  const dflash_config& c = ctx->cfg;
  const int H = c.hidden, nl = c.n_layers, ko = c.n_heads * c.head_dim, F = c.ffn;
  if (!sites) {
    ctx->conv_on = false;
    return DFLASH_OK;
  }
  if (rank < 8 || rank > kConvMaxRank || rank % 8 != 0)
    return fail(ctx, DFLASH_EINVAL, "conv rank must be a multiple of 8 in [8, 128]");
  if (H % 128 != 0) return fail(ctx, DFLASH_EINVAL, "the two-tap convolutions need hidden % 128 == 0");
  for (int i = 0; i < 4 * nl; ++i) {
    const dflash_conv_site& cs = sites[i];
    if (!cs.base || !cs.u || !cs.v) return fail(ctx, DFLASH_EINVAL, "a conv site has a NULL array");
    if (!aligned16(cs.base) || !aligned16(cs.u) || !aligned16(cs.v))
      return fail(ctx, DFLASH_EINVAL, "conv arrays must be 16-byte aligned");
  }
  const int r2 = 2 * rank;
  const size_t rows = ctx->max_rows();
  ctx->conv_on = false;
  if (ctx->conv_alloc_rank != rank) {
    void* old[] = {ctx->conv_fold, ctx->conv_vt, ctx->conv_yp, ctx->conv_h, ctx->conv_p, ctx->conv_acc};
    for (void* p : old)
      if (p) cudaFree(p);
    ctx->conv_fold = ctx->conv_h = ctx->conv_vt = nullptr;
    ctx->conv_yp = ctx->conv_p = ctx->conv_acc = nullptr;
    ctx->conv_alloc_rank = 0;
    cudaError_t e = dalloc(&ctx->conv_fold, static_cast<size_t>(nl) * r2 * (ko + F));
    if (e == cudaSuccess) e = dalloc(&ctx->conv_vt, static_cast<size_t>(nl) * 2 * H * r2);
    if (e == cudaSuccess) e = dalloc(&ctx->conv_yp, rows * (H + r2));
    if (e == cudaSuccess) e = dalloc(&ctx->conv_h, rows * H);
    if (e == cudaSuccess) e = dalloc(&ctx->conv_p, rows * r2);
    if (e == cudaSuccess) e = dalloc(&ctx->conv_acc, 2 * rows * r2);
    if (e != cudaSuccess)
      return fail(ctx, e == cudaErrorMemoryAllocation ? DFLASH_ENOMEM : DFLASH_ECUDA,
                  std::string("conv buffers: ") + cudaGetErrorString(e));
    ctx->conv_alloc_rank = rank;
  }
  ctx->m_fold_o.assign(nl, CUtensorMap{});
  ctx->m_fold_d.assign(nl, CUtensorMap{});
  for (int l = 0; l < nl; ++l) {
    const dflash_layer_weights& L = ctx->layers[l];
    uint16_t* fo = ctx->conv_fold + static_cast<size_t>(l) * r2 * (ko + F);
    uint16_t* fd = fo + static_cast<size_t>(r2) * ko;
    CK(launch_conv_fold(sites[4 * l + 1].v, L.w_o, r2, H, ko, fo, stream));
    CK(launch_conv_fold(sites[4 * l + 3].v, L.w_down, r2, H, F, fd, stream));
    CK(launch_transpose_bf16(sites[4 * l + 0].v, r2, H, ctx->conv_vt + static_cast<size_t>(2 * l) * H * r2, stream));
    CK(launch_transpose_bf16(sites[4 * l + 2].v, r2, H, ctx->conv_vt + static_cast<size_t>(2 * l + 1) * H * r2,
                             stream));
    if (!encode_2d(&ctx->m_fold_o[l], fo, r2, ko, kWeightBoxRows) ||
        !encode_2d(&ctx->m_fold_d[l], fd, r2, F, kWeightBoxRows))
      return fail(ctx, DFLASH_ECUDA, "conv fold descriptor encode failed");
  }
  if (!encode_2d(&ctx->m_vai0, sites[0].v, r2, H, kWeightBoxRows))
    return fail(ctx, DFLASH_ECUDA, "conv V descriptor encode failed");
  CK(cudaStreamSynchronize(stream));
  ctx->conv_sites.assign(sites, sites + 4 * nl);
  ctx->conv_rank = rank;
  ctx->conv_on = true;
  return DFLASH_OK;
}

dflash_status dflash_debug_wait_timeout(dflash_ctx* ctx, int limit_us, void* stream) {
  if (!ctx || limit_us < 1 || limit_us > 2000000) return ctx ? fail(ctx, DFLASH_EINVAL, "limit_us out of range") : DFLASH_EINVAL;
  CK(launch_wait_probe(1000ull * static_cast<unsigned long long>(limit_us), ctx->d_status,
                       static_cast<cudaStream_t>(stream)));
  return DFLASH_OK;
}

dflash_status dflash_debug_last_selection(dflash_ctx* ctx, int32_t* cand_out, float* u_out, float* scores_out) {
  if (!ctx) return DFLASH_EINVAL;
  if (!ctx->last_sel_rows) return fail(ctx, DFLASH_EINVAL, "the last draft did not run the path selector");
  CK(cudaDeviceSynchronize());
  const size_t n = ctx->last_sel_rows;
  if (cand_out) CK(cudaMemcpy(cand_out, ctx->sel_cand, n * kSelK * sizeof(int32_t), cudaMemcpyDeviceToHost));
  if (u_out) CK(cudaMemcpy(u_out, ctx->sel_cand_u, n * kSelK * sizeof(float), cudaMemcpyDeviceToHost));
  if (scores_out)
    CK(cudaMemcpy(scores_out, ctx->sel_scores, n * kSelK * kSelK * sizeof(float), cudaMemcpyDeviceToHost));
  return DFLASH_OK;
}

dflash_status dflash_debug_last_draft(dflash_ctx* ctx, float* hidden_out, float* top_logit_out) {
  if (!ctx) return DFLASH_EINVAL;
  CK(cudaDeviceSynchronize());
  if (hidden_out)
    CK(cudaMemcpy(hidden_out, ctx->x, static_cast<size_t>(ctx->last_rows) * ctx->cfg.hidden * sizeof(float),
                  cudaMemcpyDeviceToHost));
  if (top_logit_out && ctx->last_draft_rows)
    CK(cudaMemcpy(top_logit_out, ctx->top_logit, static_cast<size_t>(ctx->last_draft_rows) * sizeof(float),
                  cudaMemcpyDeviceToHost));
  return DFLASH_OK;
}

dflash_status dflash_debug_gemm(const uint16_t* W, const uint16_t* X, float* Y, int N, int M, int K, int splits,
                                void* stream_v) {
  dflash_ctx* ctx = nullptr;
  if (!W || !X || !Y || N < 1 || M < 1 || K < 8 || K % 8 || splits < 0) return DFLASH_EINVAL;
  if (!aligned16(W) || !aligned16(X)) return DFLASH_EINVAL;
  if (!load_encode()) return DFLASH_ECUDA;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  int dev = 0, sms = 0;
  CK(cudaGetDevice(&dev));
  CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  const int BN = gemm_token_tile(M, N, sms);
  AMaps am;
  CUtensorMap xm;
  const int xbox = splits == 0 ? gemm_act_rows(M, N, K, sms) : BN;   // CTA pairs each load half the tokens
  if (!encode_2d(&am.m[0], W, N, K, kWeightBoxRows) || !encode_2d(&xm, X, M, K, xbox)) return DFLASH_EINVAL;
  GemmWork work;
  const int G = gemm_grid(M, N, K, splits, static_cast<size_t>(1) << 40, sms);
  work.partial_elems = static_cast<size_t>(2) * G * 128 * BN;
  work.n_tickets = ceil_div(M, BN) * ceil_div(N, 128);
  int* status = nullptr;
  CK(cudaMalloc(&work.partial, work.partial_elems * sizeof(float)));
  CK(cudaMalloc(&work.tickets, work.n_tickets * sizeof(int) + sizeof(int)));
  CK(cudaMemsetAsync(work.tickets, 0, work.n_tickets * sizeof(int) + sizeof(int), stream));
  status = work.tickets + work.n_tickets;
  GemmEpi e;
  std::memset(&e, 0, sizeof(e));
  e.kind = EPI_F32_STORE;
  e.out_f32 = Y;
  e.ld_out = N;
  e.status = status;
  CK(launch_gemm(am, stacked({N}), xm, M, N, K, splits, e, work, sms, stream));
  int st = 0;
  CK(cudaStreamSynchronize(stream));
  CK(cudaMemcpy(&st, status, sizeof(int), cudaMemcpyDeviceToHost));
  cudaFree(work.partial);
  cudaFree(work.tickets);
  if (st & kDevTimeout) return DFLASH_ETIMEOUT;
  if (st) return DFLASH_EDEVICE;
  return DFLASH_OK;
}

dflash_status dflash_debug_profile(dflash_ctx* ctx, int enable) {
  if (!ctx) return DFLASH_EINVAL;
  ctx->prof_on = enable != 0;
  return DFLASH_OK;
}

dflash_status dflash_debug_profile_read(dflash_ctx* ctx, dflash_kernel_stat* out, int n) {
  if (!ctx || (n > 0 && !out)) return DFLASH_EINVAL;
  CK(cudaDeviceSynchronize());
  for (const auto& r : ctx->prof_recs) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, ctx->prof_events[r.second], ctx->prof_events[r.second + 1]) == cudaSuccess)
      ctx->prof_acc[r.first].ms += ms;
  }
  ctx->prof_recs.clear();
  ctx->prof_next = 0;
  for (int i = 0; i < n && i < DFLASH_K_COUNT; ++i) out[i] = ctx->prof_acc[i];
  for (auto& a : ctx->prof_acc) a = dflash_kernel_stat{};
  return DFLASH_OK;
}

}  // extern "C"
