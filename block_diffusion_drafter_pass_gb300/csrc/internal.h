// internal.h - declarations shared by the runtime (runtime.cu) and the kernel
// translation units (gemm_tc.cu, attention.cu, small_ops.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dfl {

constexpr int kPage = 64;          // tokens per KV page
constexpr int kMaxBatch = 64;      // sequences per call
constexpr int kMaxBlock = 32;      // block size B
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
  EPI_ARGMAX = 5       // per activation row: argmax over n (lowest index on ties)
};

struct AMaps {
  CUtensorMap m[kMaxAMaps];
};

struct ARegions {
  int n_regions;
  int paired;                       // 1: tile t reads rows 64t.. of maps 0 and 1
  int tile_begin[kMaxAMaps + 1];    // stacked: region r covers tiles [b_r, b_{r+1})
};

struct GemmEpi {
  int kind;
  // F32_STORE / F32_ADD
  float* out_f32;
  int ld_out;
  // QKV_ROPE / SWIGLU / KV_APPEND
  uint16_t* out_q;
  uint16_t* out_k;
  uint16_t* out_v;
  uint16_t* out_act;
  int n_valid;                      // SWIGLU: F (features beyond are padding)
  int head_dim;
  int n_q_heads;
  int n_kv_heads;
  const float2* rope;               // [positions][head_dim/2] (cos, sin)
  int rope_positions;
  SeqState seqs;
  SeqMeta meta;
  // KV_APPEND
  uint16_t* pool;
  int pool_pages;
  int layer0;                       // layer of region 0
  // ARGMAX
  unsigned long long* keys;         // [M] running max keys (zero between calls)
  int* done;                        // CTA completion counter (zero between calls)
  int32_t* out_ids;                 // [M]
  float* out_logit;                 // [M] (may be null)
  int* status;
};

struct GemmWork {
  float* partial;     // split-K partials
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

// BN (token tile) the GEMM uses for M rows; the activation tensor map's box
// height must equal it.
int gemm_token_tile(int M);

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
  const uint16_t* q;         // [n_seq*B][n_q*d] bf16
  float* part_o;             // [items][rows_pad][d]
  float2* part_ml;           // [items][rows_pad] (max, sum)
  uint16_t* out;             // [n_seq*B][n_q*d] bf16
  int* status;
};

// part 0: the chunked attention kernel; part 1: the combine kernel.
cudaError_t launch_attention(const CUtensorMap& pool_map, const CUtensorMap& kblk_map, const CUtensorMap& vblk_map,
                             const AttnArgs& a, int grid, int part, cudaStream_t stream);
int attention_block_rows(int B);   // key-box height used for the block's own keys

// ----------------------------------------------------------------------------
// Small kernels
// ----------------------------------------------------------------------------
cudaError_t launch_embed_norm(const uint16_t* embed, const int32_t* anchors, int mask_id, int vocab,
                              const SeqMeta& meta, int H, const uint16_t* gain, float eps, float* x, uint16_t* h,
                              int* status, cudaStream_t s);
// skip_B > 1: drop row 0 of every block of skip_B rows (rows is then n_seq*(skip_B-1)).
cudaError_t launch_rmsnorm(const float* x, int rows, int H, const uint16_t* gain, float eps, uint16_t* out,
                           int skip_B, cudaStream_t s);
cudaError_t launch_verify(const SeqMeta& meta, SeqState st, const int32_t* drafts, const int32_t* targets,
                          int32_t* tau, int32_t* bonus, cudaStream_t s);
cudaError_t launch_fuse_advance(const SeqMeta& meta, SeqState st, int pending, cudaStream_t s);
cudaError_t launch_rows_argmax_bf16(const uint16_t* logits, int rows, int cols, int32_t* out, cudaStream_t s);

}  // namespace dfl
