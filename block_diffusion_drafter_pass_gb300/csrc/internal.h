// internal.h - declarations shared by the runtime (runtime.cu) and the kernel
// translation units (gemm_tc.cu, attention.cu, small_ops.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dfl {

// Launch with programmatic stream serialization: the kernel may start while
// the previous kernel of the stream finishes; every kernel of this library
// executes griddepcontrol.wait before it touches data another kernel wrote.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// The same, as clusters of `cluster_x` CTAs along x (the grid a multiple of it).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, unsigned cluster_x,
                               cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster_x;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

constexpr int kPage = 64;          // tokens per KV page
constexpr int kMaxBatch = 64;      // sequences per call
constexpr int kMaxBlock = 32;      // block size B
constexpr int kMaxTargetLayers = 64;   // layers of a target context

// 8-bit context pages (kv_format 1): per (layer, page, kv head) one region of
//   [K codes: 64 slots][d] | [V codes: d][64 slots] (transposed), each code
//   stored as the byte code + 128 (offset binary, so the decode needs no sign fix)
//   | [K scales: 64 slots][d/32] fp16 | [V scales: d/32][64 slots] fp16,
// 136 d bytes, regions ordered (layer, page, kv head). A scale covers 32
// consecutive values of one token's head row.
__host__ __device__ constexpr size_t q8_head_bytes(int d) { return static_cast<size_t>(136) * d; }
__host__ __device__ constexpr size_t q8_vcode_off(int d) { return static_cast<size_t>(64) * d; }
__host__ __device__ constexpr size_t q8_kscale_off(int d) { return static_cast<size_t>(128) * d; }
__host__ __device__ constexpr size_t q8_vscale_off(int d) { return static_cast<size_t>(132) * d; }
constexpr int kMaxAMaps = 12;      // weight tensor maps per GEMM launch

// device status bits (dflash_sync maps them to ETIMEOUT / EDEVICE)
enum : int { kDevTimeout = 1, kDevBounds = 2 };

// Per-call sequence metadata, passed by value to kernels.
struct SeqMeta {
  int n_seq;
  int B;                           // block size (draft / verify)
  int slot[kMaxBatch];             // sequence slot per call index
  int row0[kMaxBatch + 1];         // fuse: first feature row of each sequence
};

// Device-resident state of the sequences (owned by the context).
struct SeqState {
  int* len;          // [max_seqs] committed tokens
  int* pend;         // [max_seqs] pending (appended, unverified) tokens
  int* page_table;   // [max_seqs][pages_per_seq] page ids
  int pages_per_seq;
};

// ----------------------------------------------------------------------------
// Tensor-core GEMM: OUT^T[N, M] = W[N, K] * X[M, K]^T, W the "A" operand
// (rows of up to kMaxAMaps stacked or paired weight matrices), X the "B"
// operand (activations). Epilogues consume the fp32 accumulator tile.
// ----------------------------------------------------------------------------
enum EpiKind : int {
  EPI_F32_STORE = 0,   // out_f32[m, n] = acc
  EPI_F32_ADD = 1,     // out_f32[m, n] += acc            (residual add)
  EPI_QKV_ROPE = 2,    // regions q|k|v -> bf16, RoPE on q and k
  EPI_SWIGLU = 3,      // paired gate|up -> bf16 SiLU(g) * u
  EPI_KV_APPEND = 4,   // regions (K_l, V_l)* -> RoPE(K), write to paged pool
  EPI_ARGMAX = 5,      // per activation row: argmax over n (lowest index on ties)
  EPI_RESID = 6,       // x += acc; also bf16(x * gain) and per-tile sums of x^2 (next RMSNorm)
  EPI_NORMSRC = 7      // bf16(acc * gain) and per-tile sums of acc^2 (fusion projection)
};

struct AMaps {
  CUtensorMap m[kMaxAMaps];
};

struct ARegions {
  int n_regions;
  int paired;                       // 1: tile t reads rows 64t.. of maps 0 and 1
  int pair;                         // row-pair distance: d/2 for RoPE, 64 for gate/up (32 or 64)
  int tile_begin[kMaxAMaps + 1];    // stacked: region r covers tiles [b_r, b_{r+1})
};

// Weight descriptors are encoded with boxes of this many rows (the GEMM loads
// each 128-row tile as two 64-row halves).
constexpr int kWeightBoxRows = 64;

struct GemmEpi {
  int kind;
  // F32_STORE / F32_ADD
  float* out_f32;
  int ld_out;
  // QKV_ROPE / SWIGLU / KV_APPEND
  uint16_t* out_q;                  // [M][n_q*d]
  uint16_t* out_k;                  // [M][n_kv*d]
  uint16_t* out_v;                  // transposed: [n_seq][n_kv][d][64 slots], slot = block position
  uint16_t* out_act;
  int n_valid;                      // SWIGLU: F (features beyond are padding)
  int head_dim;
  int n_q_heads;
  int n_kv_heads;
  const float2* rope;               // [positions][head_dim/2] (cos, sin)
  int rope_positions;
  SeqState seqs;
  SeqMeta meta;
  // KV_APPEND. Pool layout per (layer, page): keys [n_kv][64 slots][d], then
  // values transposed [n_kv][d][64 slots].
  uint16_t* pool;
  int pool_pages;
  int layer0;                       // layer of region 0
  int kv_q8;                        // 1: the pool holds 8-bit pages (q8_head_bytes regions)
  int qkv_f16;                      // QKV_ROPE: q, k, v stored as fp16 (the 8-bit pages' fp16 attention)
  // ARGMAX
  unsigned long long* keys;         // [M] running max keys (zero between calls)
  int* done;                        // CTA completion counter (zero between calls)
  int32_t* out_ids;                 // [M]
  float* out_logit;                 // [M] (may be null)
  int argmax_skip_B;                // > 0: rows m % B == 0 are skipped; row i*B+j -> out i*(B-1)+j-1
  int* status;
  // RMSNorm folded into the GEMM. Consumer side: the activation rows X hold
  // bf16(x * gain); each output column m is scaled by
  // rsqrt(sum_p in_ss[p][m] * inv_hidden + eps) before the epilogue op.
  const float* in_ss;               // [in_ss_parts][in_ss_ld], null = no scaling
  int in_ss_parts, in_ss_ld;
  float inv_hidden, eps;
  // Producer side (EPI_RESID / EPI_NORMSRC).
  uint16_t* out_hg;                 // [M][ld_out] bf16(x * gain)
  const uint16_t* gain;             // [N]
  float* out_ss;                    // [n_tiles][out_ss_ld] sum of x^2 over the tile's 128 features
  int out_ss_ld;
};

struct GemmWork {
  float* partial;     // stream-K partial tiles: 2 slots of 128 x BN floats per CTA
  size_t partial_elems;
  int* tickets;       // per output tile, zero between calls
  int n_tickets;
};

// Launch the GEMM. M rows of X, N = total weight rows (sum of regions, or 2*F
// padded for paired), K the reduction length. splits = 0 picks a split-K
// factor for one wave. Returns a cudaError_t.
cudaError_t launch_gemm(const AMaps& amaps, const ARegions& regions, const CUtensorMap& xmap, int M, int N,
                        int K, int splits, const GemmEpi& epi, const GemmWork& work, int num_sms,
                        cudaStream_t stream);

// BN (token tile) the GEMM uses for M rows and N output features on num_sms
// SMs; the activation tensor map's box height must equal it.
int gemm_token_tile(int M, int N, int num_sms);
// CTAs the GEMM runs with: num_sms stream-K workers (splits = 0) or
// tiles * splits, reduced until 2 partial tiles per CTA fit partial_elems.
int gemm_grid(int M, int N, int K, int splits, size_t partial_elems, int num_sms);
// True when each 256-token tile is split over K between the two CTAs of a cluster.
bool gemm_cluster_split(int M, int N, int K, int splits, int num_sms);
// CTA pairs running cta_group::2 MMAs over 256 x 256 pair tiles: 1 = pairs
// take whole pair tiles, 2 = clusters of two pairs split one pair tile's
// k-blocks; 0 = single-CTA tiles.
int gemm_pair_mode(int M, int N, int K, int splits, int num_sms);
// Box height of the activation tensor map the GEMM reads (its token tile, or
// half of it when CTA pairs split the tokens).
int gemm_act_rows(int M, int N, int K, int num_sms);

// Row-major [rows, cols] bf16 TMA descriptor (box 64 x box_rows, 128B swizzle).
bool encode_matrix_map(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows);
// Message returned by dflash_last_error(NULL).
void set_unattached_error(const char* msg);

// ----------------------------------------------------------------------------
// Block attention (split over context chunks) + combine
// ----------------------------------------------------------------------------
struct AttnArgs {
  SeqMeta meta;
  SeqState seqs;
  int layer;
  int n_q_heads, n_kv_heads, head_dim;
  int pool_pages;
  int chunk_tiles;           // context chunk in 64-key tiles
  int items_cap;             // partial-buffer capacity in work items
  int max_chunks;            // host bound on the chunks of one (sequence, kv head) row
  int rows_pad;              // row stride of the partial buffers (>= G*B)
  int spread;                // 1: G*B <= 64, query rows spread 16 per TMEM lane quarter
  int causal;                // 1: block position j sees block keys 0..j only (target pass)
  int q8;                    // 1: context pages in the 8-bit block format
  const uint16_t* q;         // [n_seq*B][n_q*d] bf16 (RoPE applied)
  const uint16_t* pool;      // the KV pool (read directly only for L2 prefetches)
  float* part_o;             // [items][rows_pad][d]
  float2* part_ml;           // [items][rows_pad] (max, sum)
  uint16_t* out;             // [n_seq*B][n_q*d] bf16
  int* status;
};

// The attention work items each CTA runs, in order: CTA c runs records
// item[off[c]] .. item[off[c+1]-1], each (sequence << 24) | (kv head << 16) |
// chunk. The host deals them from its length bounds; a record whose chunk the
// device's lengths do not reach is skipped.
constexpr int kSchedCtas = 320;
constexpr int kSchedItems = 1536;
struct AttnSched {
  uint16_t off[kSchedCtas + 1];
  uint32_t item[kSchedItems];
};

// Tensor maps the attention kernel reads through (all bf16, 128-byte swizzle):
//   pool_k  the pool as rows of d elements: key rows of (layer, page, head)
//   pool_vt the pool as rows of 64 elements: transposed value rows [dim][slot]
//   kblk    the block's keys, 3D (d, n_kv, tokens), box (64, 1, block_rows(B))
//   vblk    the block's transposed values [seq][n_kv][d][64 slots], rows of 64
struct AttnMaps {
  CUtensorMap pool_k, pool_vt, kblk, vblk;
};

// part 0: the chunked attention kernel; part 1: the combine kernel.
cudaError_t launch_attention(const AttnMaps& maps, const AttnArgs& a, const AttnSched& sched, int grid, int part,
                             cudaStream_t stream);
int attention_block_rows(int B);   // key-box height used for the block's own keys
int attention_ctas_per_sm(int head_dim, bool q8);   // resident attention CTAs per SM

// ----------------------------------------------------------------------------
// Small kernels
// ----------------------------------------------------------------------------
// Block embedding: x (fp32), hg = bf16(x * gain), ss[m] = sum(x^2).
cudaError_t launch_embed(const uint16_t* embed, const int32_t* anchors, int mask_id, const int32_t* ids, int vocab,
                         const SeqMeta& meta, int H, const uint16_t* gain, float* x, uint16_t* hg, float* ss,
                         int* status, cudaStream_t s);
// Target pass: one layer's block keys/values appended to the pool at len + j.
cudaError_t launch_block_kv_append(const SeqMeta& meta, SeqState st, int layer, const uint16_t* kb, const uint16_t* vb,
                                   uint16_t* pool, int pool_pages, int n_kv, int d, int* status, cudaStream_t s);
// Target pass: x [M][H] fp32 -> bf16 columns col0.. of feature rows of pitch ld.
cudaError_t launch_feat_copy(const float* x, int M, int H, uint16_t* feats, int ld, int col0, cudaStream_t s);
cudaError_t launch_verify(const SeqMeta& meta, SeqState st, const int32_t* drafts, const int32_t* targets,
                          int32_t* tau, int32_t* bonus, cudaStream_t s);
cudaError_t launch_fuse_advance(const SeqMeta& meta, SeqState st, int pending, cudaStream_t s);

// Page-table entries to set, table[idx[k]] = page[k], carried in the launch's
// parameter block: no host buffer has to outlive the call, and the stream
// holds only kernels, so neither the host nor the programmatic launch chain
// waits for a copy.
constexpr int kPageUpdMax = 1000;
struct PageUpdates {
  int n;
  int idx[kPageUpdMax];
  int page[kPageUpdMax];
};
cudaError_t launch_page_updates(const PageUpdates& u, int* table, cudaStream_t s);
// One bounded mbarrier wait that nothing satisfies (failure-path check).
cudaError_t launch_wait_probe(unsigned long long limit_ns, int* status, cudaStream_t s);
cudaError_t launch_rows_argmax_bf16(const uint16_t* logits, int rows, int cols, int32_t* out, cudaStream_t s);

// ----------------------------------------------------------------------------
// Two-tap dynamic convolution (DFlash 2): one apply kernel per site, CTAs of
// kConvCols columns x 16 rows. Rows are n_seq blocks of B positions; row m's
// predecessor is m - 1 unless m % B == 0.
// Input site (out_h set): x_t = rms_scale(ss, m) * xin[m] * gin; P = P[m]
//   (times the row's scale unless p_scaled); out_h[m] = bf16(Conv(x)_m); the
//   CTAs zero `zero` ([M][2r], may be null) between them.
// Output site (out_h null): x_t = y[m][0..H), P = y[m][H..H+2r);
//   x[m] += Conv(y)_m, out_hg = bf16(x * gain), out_ss[H / kConvCols parts][m]
//   = sum over the part's columns of x^2; with vt set, pacc[m][j] (zero
//   before) += the next input site's V_next (x * gain) over the CTA's columns.
// ----------------------------------------------------------------------------
constexpr int kConvMaxRank = 128;
constexpr int kConvCols = 32;      // columns per CTA = columns per sums-of-squares part
struct ConvArgs {
  int M, H, r, B;
  const uint16_t* base;   // [2][H] bf16
  const uint16_t* U;      // [2][H][r] bf16
  // input site
  const float* xin;       // [M][H] residual stream
  const uint16_t* gin;    // [H] the RMSNorm gain
  const float* ss;        // [ss_parts][ss_ld] sums of x^2
  int ss_parts, ss_ld;
  float inv_hidden, eps;
  const float* P;         // [M][2r]
  int p_scaled;           // P already carries the RMSNorm scale
  uint16_t* out_h;        // [M][H]
  float* zero;            // [M][2r] accumulator to clear, or null
  // output site
  const float* y;         // [M][ld_y]: the sublayer output, then its 2r products with V
  int ld_y;
  float* x;               // [M][H] residual stream
  uint16_t* out_hg;       // [M][H]
  const uint16_t* gain;   // [H] the next RMSNorm's gain
  float* out_ss;          // [H/kConvCols][out_ss_ld]
  int out_ss_ld;
  const uint16_t* vt;     // [H][2r] the next input site's V, transposed (null: none)
  float* pacc;            // [M][2r] accumulator of the next input site's products
  int* status;
};
cudaError_t launch_conv_apply(const ConvArgs& a, cudaStream_t s);
size_t conv_smem_bytes(int r);   // dynamic shared memory of the apply kernel at rank r (upper bound)
// Install time: F[j][c] = sum_h V[j][h] W[h][c] (bf16, fp32 sums); transpose of a bf16 matrix.
cudaError_t launch_conv_fold(const uint16_t* V, const uint16_t* W, int J, int H, int K, uint16_t* F, cudaStream_t s);
cudaError_t launch_transpose_bf16(const uint16_t* in, int rows, int cols, uint16_t* out, cudaStream_t s);

// ----------------------------------------------------------------------------
// Path selector (DFlash 2): top-16 candidates per draft row, 16 x 16 pair
// scores per adjacent pair of positions, greedy walk per sequence.
// ----------------------------------------------------------------------------
constexpr int kSelK = 16;          // candidates per masked position
constexpr int kSelDim = 256;       // width of A, B and H
constexpr int kSelMaxSlices = 64;  // column slices of a row
constexpr int kSelSliceCols = 8192;  // columns of one slice (256 threads x 8 float4)
struct SelectArgs {
  int n_seq, B, V;
  const float* logits;            // [n_seq*B][ld] fp32, scaled logits in [0, V), H(h_t) at [h_col, h_col+256)
  int ld, h_col;
  int slices;                     // ceil(V / kSelSliceCols) <= kSelMaxSlices
  unsigned long long* part;       // [n_seq*(B-1)][slices][16] keys
  const float* table;             // [V][512] fp32: W_A E[v] | W_B E[v]
  const int32_t* anchors;         // [n_seq]
  float* scores;                  // [n_seq][B-1][16][16]
  int32_t* cand;                  // [n_seq][B-1][16]
  float* cand_u;                  // [n_seq][B-1][16]
  int32_t* next;                  // [n_seq][B-1][16] the walk's pick after each predecessor rank
  float* top_logit;               // [n_seq][B-1]
  int* tickets;                   // [n_seq], zero between launches
  int32_t* draft_ids;             // [n_seq][B-1]
  int* status;
};
cudaError_t launch_path_select(const SelectArgs& s, cudaStream_t stream);

// ----------------------------------------------------------------------------
// Temperature sampling (top-k <= 32, top-p) and the speculative-sampling verify
// ----------------------------------------------------------------------------
constexpr int kSampleWidth = 32;     // list width: ids / probabilities per row
constexpr int kSampleMaxSlices = 64; // column slices of a row
struct FilterArgs {
  const unsigned long long* part;  // [rows][slices][32] slice lists
  int slices;
  float inv_temperature;
  int top_k;                       // 1..32
  float top_p;                     // (0, 1]
  const float* uniforms;           // [rows] (with drawn)
  int32_t* out_ids;                // [rows][32], -1 past the kept entries
  float* out_probs;                // [rows][32]
  int32_t* drawn;                  // [rows] or null
};
struct VerifySampleArgs {
  const int32_t* drafts;           // [n][B-1]
  const int32_t* q_ids;            // [n][B-1][32] the drafter's filtered lists
  const float* q_probs;
  const int32_t* p_ids;            // [n][B][32] the target's filtered lists
  const float* p_probs;
  const float* u_accept;           // [n][B-1]
  const float* u_resample;         // [n][B]
  int32_t* tau;                    // [n]
  int32_t* bonus;                  // [n]
  int* status;
};
// Slice lists (topk_slices_kernel, 32 wide) then the filter / draw of every
// row. bf16: rows of a [rows][ld] bf16 matrix; otherwise fp32 rows of the
// drafter's logits with the block's anchor rows skipped (draft_B = B).
cudaError_t launch_sample_filter(const void* logits, bool bf16, int ld, int V, int rows, int draft_B,
                                 unsigned long long* part, const FilterArgs& fa, cudaStream_t s);
int sample_slice_cols(bool bf16);
cudaError_t launch_verify_sample(const SeqMeta& meta, SeqState st, const VerifySampleArgs& a, cudaStream_t s);

}  // namespace dfl
