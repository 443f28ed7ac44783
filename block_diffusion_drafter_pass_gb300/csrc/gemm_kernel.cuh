// gemm_kernel.cuh - the drafter's dense contractions on the 5th-generation tensor
// cores (tcgen05.mma, fp32 accumulators in TMEM, operands staged by TMA).
//
// Every projection of the drafter pass is OUT^T[N, M] = W[N, K] * X[M, K]^T:
// the weight rows are the UMMA "A" operand (M_mma = 128 rows per tile) and
// the tokens the "B" operand (N_mma = BN, 16..256), so a batch-1 block of 16
// tokens still fills the 128-row tensor-core tile and the kernel streams
// weights at HBM speed; with 512 tokens the same kernel is compute bound.
//
// Persistent stream-K: one CTA per SM streams an equal, contiguous range of
// (tile, 64-wide k-block) units through a STAGES-deep TMA ring. CTA = 6 warps:
// warp 0 issues the TMA loads, warp 1 owns TMEM and issues the MMAs (one
// thread) into one of two accumulator buffers, warps 2-5 drain the other
// buffer (tcgen05.ld) and run the fused epilogue:
//   EPI_F32_STORE  plain fp32 output (tests)
//   EPI_RESID      x += acc, then bf16(x * g) and sum(x^2) for the next RMSNorm
//   EPI_NORMSRC    bf16(acc * g) and sum(acc^2) (fusion projection W_c)
//   EPI_QKV_ROPE   q/k/v split with rotate-half RoPE on q and k
//   EPI_SWIGLU     SiLU(gate) * up from paired gate/up weight rows
//   EPI_KV_APPEND  KV injection: RoPE(W_K H_t), W_V H_t scattered to pages
//   EPI_ARGMAX     LM head with the per-row argmax fused; logits never stored
// A tile split over several CTAs is finished by the last one to arrive (an
// atomic ticket; nothing spins): it adds the others' partial tiles to its own
// accumulator and runs the epilogue.
//
// RoPE and SwiGLU pair tile row r with row r ^ P (P = d/2 for RoPE, 64 for
// gate/up rows); those live in another warp's TMEM lanes, so the pair is
// exchanged through a double-buffered shared-memory stage, one named barrier
// per 16-column chunk.
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace dfl {
namespace gk {

// Epilogue classes: each kernel instantiation carries the code of one class
// only, so the kind is a compile-time constant (or one of two) and the
// chunk loop stays small.
enum : int { kEcF32 = 0, kEcNorm = 1, kEcRope = 2, kEcSwiglu = 3, kEcArgmax = 4 };

__host__ __device__ constexpr int epilogue_class(int kind) {
  return kind == EPI_RESID || kind == EPI_NORMSRC       ? kEcNorm
         : kind == EPI_QKV_ROPE || kind == EPI_KV_APPEND ? kEcRope
         : kind == EPI_SWIGLU                            ? kEcSwiglu
         : kind == EPI_ARGMAX                            ? kEcArgmax
                                                         : kEcF32;
}

// The run-time kind narrowed to the kinds of class EC.
template <int EC>
__device__ __forceinline__ int class_kind(int kind) {
  if constexpr (EC == kEcNorm) return kind == EPI_NORMSRC ? EPI_NORMSRC : EPI_RESID;
  else if constexpr (EC == kEcRope) return kind == EPI_KV_APPEND ? EPI_KV_APPEND : EPI_QKV_ROPE;
  else if constexpr (EC == kEcSwiglu) return EPI_SWIGLU;
  else if constexpr (EC == kEcArgmax) return EPI_ARGMAX;
  else return kind == EPI_F32_ADD ? EPI_F32_ADD : EPI_F32_STORE;
}

constexpr int kThreads = 192;
constexpr int kTileN = 128;     // weight rows per tile (UMMA M)
constexpr int kTileK = 64;      // K per stage (one 128-byte swizzle row)
constexpr int kABytes = kTileN * kTileK * 2;

template <int BN>
struct Cfg {
  static constexpr int kBBytes = BN * kTileK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = BN <= 64 ? 8 : (BN <= 128 ? 6 : 4);
  static constexpr int kTmemCols = 2 * BN < 32 ? 32 : 2 * BN;     // two accumulator buffers
  static constexpr int kStgBytes = 2 * 128 * 17 * 4;                // pair-exchange stage (x2)
  static constexpr int kSmem = kStages * kStageBytes + kStgBytes + 1024;
};

struct GemmArgs {
  int M, N, K;
  int k_blocks, n_tiles, m_tiles;
  long long units;     // tiles * k_blocks
  int grid;            // CTAs
  int workers;         // stream-K workers: CTAs, or CTA pairs (pair = 3)
  int csplit;          // 1: CTAs 2t and 2t+1 form a cluster splitting tile t's k-blocks in halves
  int pair;            // 1: CTA pairs run cta_group::2 MMAs over whole 256 x 256 pair tiles;
                       // 2: clusters of two such pairs, each over half of the k-blocks of one pair tile;
                       // 3: CTA pairs over equal ranges of (pair tile, k-block) units (stream-K)
  float* partial;      // [grid][2][128 * BN] partial tiles
  int* tickets;        // [tiles], zero between launches
  int* status;
};

// Named barriers of the epilogue warps: barrier 1 + grp joins the 128 threads
// of epilogue group grp (one warp per TMEM lane quarter); barrier 3 joins the
// 256 threads of both groups of the pair kernel.
__device__ __forceinline__ void epi_bar(int grp = 0) { asm volatile("bar.sync %0, 128;" ::"r"(1 + grp) : "memory"); }
__device__ __forceinline__ void epi_bar_all() { asm volatile("bar.sync 3, 256;" ::: "memory"); }

// Reductions over the tile's 128 rows go through shared memory: a 16-column
// chunk is staged as [128 rows][17], thread t reduces rows 16*(t>>4) .. +15
// of column t&15, and 16 threads combine the 8 row groups.
struct EpiShared {
  union {   // one kernel instantiation uses one of them; slot = epilogue group * 2 + chunk parity
    unsigned long long cand8[4][8][16];  // argmax candidate per (row group, column)
    float red8[4][8][16];                // sum of squares per (row group, column)
  };
  int row_pos[256];                  // QKV_ROPE / KV_APPEND: absolute position of each column
  int row_dst[256];                  // KV_APPEND: (page, slot) part of the pool row index
  float row_scale[256];              // folded RMSNorm scale of each column
  float2 rope_base[16][64];          // RoPE (cos, sin) at each chunk's first position, per frequency
  int flag[2];                       // per epilogue group
};

__device__ __forceinline__ int region_of(const ARegions& rg, int tile) {
  int r = 0;
  while (r + 1 < rg.n_regions && tile >= rg.tile_begin[r + 1]) ++r;
  return r;
}

// TMA sources of the tile's two 64-row halves: stacked regions read 128
// consecutive rows of one matrix; paired tiles read 64 gate rows and the same
// 64 up rows.
__device__ __forceinline__ void weight_rows(const ARegions& rg, int tile_n, int& map_lo, int& row_lo, int& map_hi,
                                            int& row_hi) {
  if (rg.paired) {
    map_lo = 0;
    map_hi = 1;
    row_lo = row_hi = tile_n * 64;
  } else {
    const int reg = region_of(rg, tile_n);
    map_lo = map_hi = reg;
    row_lo = (tile_n - rg.tile_begin[reg]) * kTileN;
    row_hi = row_lo + 64;
  }
}

__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// Folded RMSNorm scale of activation row m: 8 independent partial loads per
// batch so the sum costs a few memory latencies, not one per partial.
__device__ __forceinline__ float norm_scale(const GemmEpi& e, int m) {
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  int p = 0;
  for (; p + 8 <= e.in_ss_parts; p += 8) {
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[q] += __ldcg(e.in_ss + static_cast<size_t>(p + q) * e.in_ss_ld + m);
  }
  for (; p < e.in_ss_parts; ++p) acc[0] += __ldcg(e.in_ss + static_cast<size_t>(p) * e.in_ss_ld + m);
  const float ss = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
  return rsqrtf(ss * e.inv_hidden + e.eps);
}

// Per-column metadata of one output tile (columns m0 .. m0+BN-1), computed
// once by all 128 epilogue threads before the tile is drained.
// Columns [cb, ce) of the tile, by epilogue group grp.
template <int BN, int EC>
__device__ __forceinline__ void tile_cols_prepare(const GemmArgs& a, const GemmEpi& e, int m0, int r,
                                                  EpiShared& sh, int cb = 0, int ce = BN, int grp = 0) {
  const int kind = class_kind<EC>(e.kind);
  for (int col = cb + r; col < ce; col += 128) {
    const int m = m0 + col;
    float sc = 1.f;
    int pos = -1, dst = -1;
    if (m < a.M) {
      if (e.in_ss) sc = norm_scale(e, m);
      if (kind == EPI_QKV_ROPE) {
        const int i = m / e.meta.B, j = m - i * e.meta.B;
        pos = e.seqs.len[e.meta.slot[i]] + j;
      } else if (kind == EPI_KV_APPEND) {
        int i = 0;
        while (i + 1 < e.meta.n_seq && m >= e.meta.row0[i + 1]) ++i;
        const int slot = e.meta.slot[i];
        pos = e.seqs.len[slot] + e.seqs.pend[slot] + (m - e.meta.row0[i]);
        const int pg_idx = pos / kPage;
        if (pg_idx < e.seqs.pages_per_seq) {
          const int page = e.seqs.page_table[static_cast<size_t>(slot) * e.seqs.pages_per_seq + pg_idx];
          if (page >= 0 && page < e.pool_pages) dst = page * 2 * e.n_kv_heads * kPage + (pos % kPage);
        }
        if (dst < 0) latch_status(e.status, kDevBounds);
      }
      if (pos >= e.rope_positions) {
        latch_status(e.status, kDevBounds);
        pos = -1;
        dst = -1;
      }
    }
    sh.row_scale[col] = sc;
    sh.row_pos[col] = pos;
    sh.row_dst[col] = dst;
  }
  epi_bar(grp);
  // RoPE bases of every chunk: one round of loads for the whole column range
  if (kind == EPI_QKV_ROPE || kind == EPI_KV_APPEND) {
    const int half = e.head_dim >> 1;
    for (int k = r; k < ((ce - cb) / 16) * half; k += 128) {
      const int kc = k / half, fi = k - kc * half, ch = cb / 16 + kc;
      const int pos = sh.row_pos[ch * 16];
      sh.rope_base[ch][fi] = pos >= 0 ? e.rope[static_cast<size_t>(pos) * half + fi] : make_float2(1.f, 0.f);
    }
    epi_bar(grp);
  }
}

// 32 consecutive TMEM columns of this thread's lane (32x32b shape);
// completes with tcgen05.wait::st.
__device__ __forceinline__ void tmem_store32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]), "f"(v[8]),
      "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]), "f"(v[15]), "f"(v[16]),
      "f"(v[17]), "f"(v[18]), "f"(v[19]), "f"(v[20]), "f"(v[21]), "f"(v[22]), "f"(v[23]), "f"(v[24]),
      "f"(v[25]), "f"(v[26]), "f"(v[27]), "f"(v[28]), "f"(v[29]), "f"(v[30]), "f"(v[31])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st_gk() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Residual inputs of one 16-column chunk (EPI_RESID); the chunk loop keeps
// them two chunks ahead of use.
// LM head: after a tile's epilogue, the CTA that finishes the last of
// `total` tile epilogues decodes the winning keys into ids (and logits) and
// resets them for the next call.
__device__ __forceinline__ void argmax_tile_done(const GemmArgs& a, const GemmEpi& e, EpiShared& esh, int r,
                                                 int total, int grp = 0) {
  __threadfence();
  epi_bar(grp);
  if (r == 0) {
    const int dn = atomicAdd(e.done, 1);
    esh.flag[grp] = (dn == total - 1);
  }
  epi_bar(grp);
  if (esh.flag[grp]) {
    __threadfence();
    const int sb = e.argmax_skip_B;
    for (int m = r; m < a.M; m += 128) {
      if (sb > 0 && m % sb == 0) continue;
      const int o = sb > 0 ? (m / sb) * (sb - 1) + (m % sb) - 1 : m;
      const unsigned long long k = atomicExch(e.keys + m, 0ull);
      e.out_ids[o] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(k & 0xFFFFFFFFull));
      if (e.out_logit) {
        const float raw = ordered_key_inv(static_cast<uint32_t>(k >> 32));
        e.out_logit[o] = e.in_ss ? raw * norm_scale(e, m) : raw;
      }
    }
    if (r == 0) *e.done = 0;
  }
  epi_bar(grp);
}

// Stream-K partition: worker g (a CTA, or a CTA pair) owns the contiguous
// range of (tile, k-block) units [unit_begin(g), unit_begin(g + 1)); tiles are
// ordered so that the m tiles of one weight tile are consecutive (weights
// reused from L2).
// floor(x / y) for x >= 0, y > 0; a 32-bit division whenever both fit
// (a 64-bit division is a long dependent instruction sequence)
__device__ __forceinline__ long long div_floor(long long x, long long y) {
  if (((x | y) >> 32) == 0) return static_cast<long long>(static_cast<uint32_t>(x) / static_cast<uint32_t>(y));
  return x / y;
}
__device__ __forceinline__ long long unit_begin(int g, const GemmArgs& a) {
  return div_floor(static_cast<long long>(g) * a.units, a.workers);
}
// The worker whose range holds unit u: the largest g with floor(g U / G) <= u,
// i.e. g U < (u + 1) G, which is floor(((u + 1) G - 1) / U).
__device__ __forceinline__ int cta_of(long long u, const GemmArgs& a) {
  return static_cast<int>(div_floor((u + 1) * a.workers - 1, a.units));
}

__device__ __forceinline__ void load_resid(const GemmArgs& a, const GemmEpi& e, int m0, int c0, int n,
                                           float (&x)[16]) {
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    const int m = m0 + c0 + c;
    x[c] = (n < a.N && m < a.M && c0 < a.M) ? __ldcg(e.out_f32 + static_cast<size_t>(m) * e.ld_out + n) : 0.f;
  }
}

// Partial tiles hold column runs of four: value (column c, row r) sits at
// float ((c / 4) * 128 + r) * 4 + c % 4 of the slot, so a row's four columns
// are one 16-byte access and a warp's access covers 512 contiguous bytes.
// part_row(slot, r) is row r's first run; run j is 512 floats further.
constexpr int kPartRun = kTileN * 4;
__device__ __forceinline__ float* part_row(float* slot, int r) { return slot + 4 * r; }
__device__ __forceinline__ const float* part_row(const float* slot, int r) { return slot + 4 * r; }

// 16 partial values of one row: columns c0 .. c0 + 15 (c0 a multiple of 4).
__device__ __forceinline__ void part_load16(const float* row, int c0, float (&v)[16]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float4 t = __ldcg(reinterpret_cast<const float4*>(row + static_cast<size_t>((c0 >> 2) + j) * kPartRun));
    v[4 * j] = t.x;
    v[4 * j + 1] = t.y;
    v[4 * j + 2] = t.z;
    v[4 * j + 3] = t.w;
  }
}

// Park a tile's partial sum: TMEM columns [cb, ce) of this thread's lane to
// its row of the slot (row = part_row(slot, lane)), 16 or 32 columns per TMEM load.
template <int BN>
__device__ __forceinline__ void park_partial(uint32_t tb, float* row, int cb = 0, int ce = BN) {
  if constexpr (BN < 32) {
#pragma unroll
    for (int c0 = cb; c0 < ce; c0 += 16) {
      float v[16];
      tmem_ld16(tb + c0, v);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        *reinterpret_cast<float4*>(row + static_cast<size_t>((c0 >> 2) + j) * kPartRun) =
            make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    }
  } else {
#pragma unroll 1
    for (int c0 = cb; c0 < ce; c0 += 32) {
      float v[32];
      tmem_ld32(tb + c0, v);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        *reinterpret_cast<float4*>(row + static_cast<size_t>((c0 >> 2) + j) * kPartRun) =
            make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    }
  }
}

// Per-lane epilogue inputs read from memory that do not depend on the
// accumulator: the row's RMSNorm gain (RESID, NORMSRC) and its RoPE rotation
// (the table's position 1). Read before the accumulator wait, so their
// latency overlaps the MMAs instead of opening the epilogue.
struct EpiPre {
  float gain;
  float2 rot;
};

template <int EC>
__device__ __forceinline__ EpiPre epi_pre(const GemmArgs& a, const ARegions& rg, const GemmEpi& e, int tile, int r) {
  EpiPre p;
  p.gain = 0.f;
  p.rot = make_float2(1.f, 0.f);
  const int kind = class_kind<EC>(e.kind);
  const int tn = tile / a.m_tiles;
  if (kind == EPI_RESID || kind == EPI_NORMSRC) {
    const int n = tn * kTileN + r;
    if (n < a.N) p.gain = bf16_to_f32(e.gain[n]);
  } else if (kind == EPI_QKV_ROPE || kind == EPI_KV_APPEND) {
    int reg = 0, rf = r;
    if (!rg.paired) {
      reg = region_of(rg, tn);
      rf = (tn - rg.tile_begin[reg]) * kTileN + r;
    }
    const bool rope = kind == EPI_QKV_ROPE ? reg < 2 : (reg & 1) == 0;
    if (rope) {
      const int d = e.head_dim > 0 ? e.head_dim : 1, half = d >> 1;
      const int di = rf % d;
      p.rot = e.rope[half + ((r & rg.pair) == 0 ? di : di - half)];
    }
  }
  return p;
}

// Stores one 16-token chunk of bf16 rows whose 128 tile rows are contiguous
// features of each token's output row (q / k rows, the keys of a page slot):
// each thread puts its row's 16 values into a free 128 x 16 staging buffer
// (token-major), and after a barrier writes 32 contiguous bytes of one
// token, so a warp writes four tokens' 256-byte runs instead of sixteen
// 64-byte pieces. dst(token) is the token's first output element for tile
// row 0 (rows of one head stay within 16-row segments), or null to skip it.
// Ends with a barrier, so the buffer can be reused.
template <typename Dst>
__device__ __forceinline__ void store_chunk_transposed(const uint16_t (&ov)[16], int r, float* buf, int grp, Dst dst) {
  uint16_t* t = reinterpret_cast<uint16_t*>(buf);
#pragma unroll
  for (int c = 0; c < 16; ++c) t[c * 128 + r] = ov[c];
  epi_bar(grp);
  const int c = r >> 3, seg = (r & 7) * 16;
  uint16_t* p = dst(c, seg);
  if (p) {
    const uint4* src = reinterpret_cast<const uint4*>(t + c * 128 + seg);
    reinterpret_cast<uint4*>(p)[0] = src[0];
    reinterpret_cast<uint4*>(p)[1] = src[1];
  }
  epi_bar(grp);
}

// Drain one finished tile from TMEM (plus the other workers' partial tiles)
// and run the epilogue. r = TMEM lane of this thread (0..127). g, first and
// last are stream-K workers; worker w's partial slots belong to CTA
// w * cstep + cbase (CTA pairs: the pair's CTA that holds the same weight
// tile), and tile_u0 is the tile's first unit in the workers' partition.
// G = 2: two epilogue groups each drain a column range [cbeg, cend) of the
// tile; group grp has its own named barrier, staging buffer (single-buffered,
// with one more barrier per chunk where rows are exchanged) and reduction
// slots.
template <int BN, int EC, int G = 1>
__device__ __forceinline__ void epilogue_tile(const GemmArgs& a, const ARegions& rg, const GemmEpi& e, int g,
                                              int tile, int first, int last, uint32_t tb, int r, EpiShared& sh,
                                              float* stg, uint32_t pre, const float (&rpre)[16], const EpiPre& pp,
                                              int cbeg, int cend, const float* speer, long long tile_u0,
                                              int cstep = 1, int cbase = 0, int grp = 0) {
  const int kind = class_kind<EC>(e.kind);
  const int q = r >> 5, lane = r & 31;
  const int tn = tile / a.m_tiles, tm = tile - tn * a.m_tiles;
  const int m0 = tm * BN;
  const int P = rg.pair;
  const int f = r;                              // row of this lane within the tile
  const size_t slot_elems = static_cast<size_t>(kTileN) * BN;

  // kind-specific constants of this lane
  int reg = 0, rf = f;                          // region and row within the region's matrix
  if (!rg.paired) {
    reg = region_of(rg, tn);
    rf = (tn - rg.tile_begin[reg]) * kTileN + f;
  }
  const int n = tn * kTileN + f;                // output feature (plain kinds)
  const int d = e.head_dim > 0 ? e.head_dim : 1, half = d >> 1;
  const int hd = rf / d, di = rf - hd * d;
  const bool lo = (r & P) == 0;                 // lower member of the row pair (r, r ^ P)
  const bool paired_kind = kind == EPI_SWIGLU || kind == EPI_QKV_ROPE || kind == EPI_KV_APPEND;
  bool rope = false;
  if (kind == EPI_QKV_ROPE) rope = reg < 2;
  if (kind == EPI_KV_APPEND) rope = (reg & 1) == 0;
  const int fi = lo ? di : di - half;           // RoPE frequency index of the pair
  const float gain = pp.gain;

  // Other CTAs holding partial sums of this tile. A one-chunk tile reads up
  // to kRound of them in one round of loads; wider tiles read one a chunk
  // ahead into registers. Any further pieces are read on use. The pieces are
  // added in CTA order whichever CTA finishes the tile, so the result is the
  // same from run to run. Every CTA after the tile's first one starts inside
  // the tile, so its piece is its first segment (slot 0); the first CTA's
  // piece is in slot 1 when that CTA began in an earlier tile.
  const bool first_in_slot1 = unit_begin(first, a) < tile_u0;
  auto partial_src = [&](int o) {
    const int side = (o == first && first_in_slot1) ? 1 : 0;
    return part_row(a.partial + (static_cast<size_t>(o * cstep + cbase) * 2 + side) * slot_elems, r);
  };
  // wider tiles: the first kAhead other pieces, in CTA order, are read one
  // chunk ahead, all in one round of loads (256-token tiles: two, the most a
  // stream-K pair range splits a tile into when it holds more than one
  // tile's units; further pieces are read on use)
  constexpr int kAhead = BN >= 256 ? 2 : 3;
  const float* psrc[kAhead];
#pragma unroll
  for (int k = 0; k < kAhead; ++k) {   // the k-th other piece: worker first + k, skipping g
    const int o = first + k + (first + k >= g ? 1 : 0);
    psrc[k] = o <= last ? partial_src(o) : nullptr;
  }
  const int n_oth = last - first;
  auto partial_load = [&](int c0, float (&p0)[kAhead][16]) {
#pragma unroll
    for (int k = 0; k < kAhead; ++k) {
      if (psrc[k]) {
        part_load16(psrc[k], c0, p0[k]);
      } else {
#pragma unroll
        for (int c = 0; c < 16; ++c) p0[k][c] = 0.f;
      }
    }
  };
  // RoPE: when a chunk's 16 positions are consecutive (one sequence's block),
  // (cos, sin) is read once at its first position and advanced by the row's
  // rotation R = (cos, sin) of its frequency (the table's position 1) with a
  // complex multiply per column; otherwise it is read per column.
  const bool resid = kind == EPI_RESID;
  float ra[16], rb[16];
  float2 rot = make_float2(1.f, 0.f);
  // pre != 0: the residual tile already sits in TMEM at `pre` (loaded while
  // the MMAs ran); otherwise it is read two chunks ahead
  if (resid && !pre) {
    if constexpr (BN == 16) {
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        ra[c] = rpre[c];
        rb[c] = 0.f;
      }
    } else {
      load_resid(a, e, m0, cbeg, n, ra);
      load_resid(a, e, m0, cbeg + 16, n, rb);
    }
  }
  if (rope) rot = pp.rot;
  float pc0[kAhead][16];
  if constexpr (BN > 16) {
    if (n_oth) partial_load(cbeg, pc0);
  }
#pragma unroll 1
  for (int c0 = cbeg; c0 < cend; c0 += 16) {
    const int buf = (c0 >> 4) & 1;
    float* sb = G == 1 ? stg + buf * (128 * 17) : stg + grp * (128 * 17);
    const int pb = buf + 2 * grp;   // reduction slot of this chunk
    float rc[16];
    if (resid && !pre && c0 + 32 < cend) load_resid(a, e, m0, c0 + 32, n, rc);
    float rx[16];
    if (resid) {
      if (pre) {
        tmem_ld16(pre + c0, rx);
      } else {
#pragma unroll
        for (int c = 0; c < 16; ++c) rx[c] = ra[c];
      }
    }
    float pn0[kAhead][16];
    if constexpr (BN > 16) {
      if (n_oth && c0 + 16 < cend) partial_load(c0 + 16, pn0);
    }
    float v[16];
    tmem_ld16(tb + c0, v);
    if (speer) {   // the cluster peer's half-K sum of these columns, [column - cbeg][row]
#pragma unroll
      for (int c = 0; c < 16; ++c) v[c] += speer[(c0 - cbeg + c) * 128 + r];
    }
    constexpr int kRound = 7;
    if (BN == 16 && first != last && last - first <= kRound) {
      // the other pieces in CTA order: k-th other CTA is first + k, skipping g
      float pv[kRound][16];
#pragma unroll
      for (int k = 0; k < kRound; ++k) {
        const int o = first + k + (first + k >= g ? 1 : 0);
        if (o <= last) {
          part_load16(partial_src(o), 0, pv[k]);
        } else {
#pragma unroll
          for (int c = 0; c < 16; ++c) pv[k][c] = 0.f;
        }
      }
      float sum[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) sum[c] = 0.f;
#pragma unroll
      for (int p = 0; p <= kRound; ++p) {
        const int o = first + p;
        if (o <= last) {
          // position p is this CTA's own piece, or other piece p (before g) or p - 1 (after g)
#pragma unroll
          for (int c = 0; c < 16; ++c)
            sum[c] += o == g ? v[c] : (o < g ? pv[p < kRound ? p : kRound - 1][c] : pv[p > 0 ? p - 1 : 0][c]);
        }
      }
#pragma unroll
      for (int c = 0; c < 16; ++c) v[c] = sum[c];
    } else if (first != last) {
      float sum[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) sum[c] = 0.f;
      for (int o = first; o <= last; ++o) {
        const int k = (o - first) - (o > g ? 1 : 0);   // rank of o among the other pieces
        if (o == g) {
#pragma unroll
          for (int c = 0; c < 16; ++c) sum[c] += v[c];
        } else if (BN > 16 && k < kAhead) {
#pragma unroll
          for (int kk = 0; kk < kAhead; ++kk) {
            if (kk == k) {
#pragma unroll
              for (int c = 0; c < 16; ++c) sum[c] += pc0[kk][c];
            }
          }
        } else {
          float pv[16];
          part_load16(partial_src(o), c0, pv);
#pragma unroll
          for (int c = 0; c < 16; ++c) sum[c] += pv[c];
        }
      }
#pragma unroll
      for (int c = 0; c < 16; ++c) v[c] = sum[c];
    }
    if (e.in_ss && kind != EPI_ARGMAX) {
#pragma unroll
      for (int c = 0; c < 16; ++c) v[c] *= sh.row_scale[c0 + c];
    }
    float other[16];
    if (paired_kind) {   // exchange with row r ^ P through the chunk's staging buffer
#pragma unroll
      for (int c = 0; c < 16; ++c) sb[r * 17 + c] = v[c];
      epi_bar(grp);
      const int pr = r ^ P;
#pragma unroll
      for (int c = 0; c < 16; ++c) other[c] = sb[pr * 17 + c];
      if constexpr (G == 2) epi_bar(grp);   // single buffer: all reads before the next chunk's writes
    }

    if (kind == EPI_F32_STORE || kind == EPI_F32_ADD) {
      if (n < a.N && m0 + c0 + 16 <= a.M) {
        float* p = e.out_f32 + static_cast<size_t>(m0 + c0) * e.ld_out + n;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          if (kind == EPI_F32_ADD) *p += v[c]; else *p = v[c];
          p += e.ld_out;
        }
      } else if (n < a.N) {
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const int m = m0 + c0 + c;
          if (m < a.M) {
            float* p = e.out_f32 + static_cast<size_t>(m) * e.ld_out + n;
            if (kind == EPI_F32_ADD) *p += v[c]; else *p = v[c];
          }
        }
      }
    } else if (kind == EPI_RESID || kind == EPI_NORMSRC) {
      if (n < a.N && m0 + c0 + 16 <= a.M) {   // whole chunk: pointers advance by the row stride
        const size_t ld = e.ld_out;
        float* px = e.out_f32 + static_cast<size_t>(m0 + c0) * ld + n;
        uint16_t* ph = e.out_hg + static_cast<size_t>(m0 + c0) * ld + n;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          float xn = v[c];
          if (kind == EPI_RESID) {
            xn += rx[c];
            *px = xn;
            px += ld;
          }
          *ph = f32_to_bf16(xn * gain);
          ph += ld;
          sb[r * 17 + c] = xn * xn;
        }
      } else {
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const int m = m0 + c0 + c;
          float xn = 0.f;
          if (n < a.N && m < a.M) {
            const size_t off = static_cast<size_t>(m) * e.ld_out + n;
            xn = v[c];
            if (kind == EPI_RESID) {
              xn += rx[c];
              e.out_f32[off] = xn;
            }
            e.out_hg[off] = f32_to_bf16(xn * gain);
          }
          sb[r * 17 + c] = xn * xn;
        }
      }
      // column sums of squares over the tile's 128 rows
      epi_bar(grp);
      const int cc = r & 15, gq = r >> 4;
      float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < 16; ++i) s4[i & 3] += sb[(gq * 16 + i) * 17 + cc];
      sh.red8[pb][gq][cc] = (s4[0] + s4[1]) + (s4[2] + s4[3]);
      epi_bar(grp);
      if (r < 16) {
        const int m = m0 + c0 + r;
        float t = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) t += sh.red8[pb][k][r];
        if (m < a.M) e.out_ss[static_cast<size_t>(tn) * e.out_ss_ld + m] = t;
      }
    } else if (kind == EPI_ARGMAX) {
      // per column: highest logit over the tile's rows, lowest row on ties,
      // packed as (ordered key << 32) | ~row so one 64-bit max decides
#pragma unroll
      for (int c = 0; c < 16; ++c) sb[r * 17 + c] = v[c];
      epi_bar(grp);
      const int cc = r & 15, gq = r >> 4;
      const int m = m0 + c0 + cc;
      unsigned long long best = 0ull;
      if (m < a.M && !(e.argmax_skip_B > 0 && m % e.argmax_skip_B == 0)) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int row = gq * 16 + i;
          const uint32_t idx = static_cast<uint32_t>(tn * kTileN + row);
          const float lv = sb[row * 17 + cc];
          const unsigned long long cand =   // -0 and +0 are one value, as in a float argmax
              (static_cast<unsigned long long>(ordered_key(lv == 0.f ? 0.f : lv)) << 32) | (0xFFFFFFFFu - idx);
          best = (static_cast<int>(idx) < a.N && cand > best) ? cand : best;
        }
      }
      sh.cand8[pb][gq][cc] = best;
      epi_bar(grp);
      if (r < 16) {
        unsigned long long b8 = sh.cand8[pb][0][r];
#pragma unroll
        for (int k = 1; k < 8; ++k) b8 = sh.cand8[pb][k][r] > b8 ? sh.cand8[pb][k][r] : b8;
        if (b8) atomicMax(e.keys + (m0 + c0 + r), b8);
      }
    } else if (kind == EPI_SWIGLU) {
      // rows < 64 hold gate rows, rows >= 64 the up rows of the same features;
      // each member of a pair writes half of the columns
      const int fint = tn * 64 + (f & 63);
      if (fint < e.n_valid && m0 + c0 + 16 <= a.M) {   // whole chunk
        const size_t ld = e.n_valid;
        uint16_t* p = e.out_act + static_cast<size_t>(m0 + c0 + (lo ? 0 : 8)) * ld + fint;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const float gt = lo ? v[c] : other[c + 8], up = lo ? other[c] : v[c + 8];
          *p = f32_to_bf16(silu_f(gt) * up);
          p += ld;
        }
      } else {
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const int m = m0 + c0 + c;
          if ((c < 8) == lo && fint < e.n_valid && m < a.M) {
            const float gt = lo ? v[c] : other[c], up = lo ? other[c] : v[c];
            e.out_act[static_cast<size_t>(m) * e.n_valid + fint] = f32_to_bf16(silu_f(gt) * up);
          }
        }
      }
    } else if (kind == EPI_QKV_ROPE && reg == 2 && e.meta.B % 16 == 0 && m0 + c0 + 16 <= a.M &&
               sh.row_pos[c0] >= 0 && sh.row_pos[c0 + 15] >= 0) {
      // values, transposed: the chunk's 16 tokens are 16 consecutive slots of
      // one sequence, written as two 16-byte stores
      const int i = (m0 + c0) / e.meta.B, j0 = (m0 + c0) - i * e.meta.B;
      uint32_t w[8];
      const bool h16 = e.qkv_f16 != 0;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint32_t lo = h16 ? f32_to_f16(v[2 * c]) : f32_to_bf16(v[2 * c]);
        const uint32_t hi = h16 ? f32_to_f16(v[2 * c + 1]) : f32_to_bf16(v[2 * c + 1]);
        w[c] = lo | (hi << 16);
      }
      uint4* dstv = reinterpret_cast<uint4*>(
          e.out_v + ((static_cast<size_t>(i) * e.n_kv_heads + hd) * d + di) * kPage + j0);
      dstv[0] = make_uint4(w[0], w[1], w[2], w[3]);
      dstv[1] = make_uint4(w[4], w[5], w[6], w[7]);
    } else {   // EPI_QKV_ROPE or EPI_KV_APPEND
      // Every shared-memory input of the chunk is read, and every output
      // value computed, before the chunk's first global store: loads placed
      // after a store would wait for it.
      int posv[16], dstv[16];
      bool allpos = true, alldst = true;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        posv[c] = sh.row_pos[c0 + c];
        dstv[c] = kind == EPI_KV_APPEND ? sh.row_dst[c0 + c] : 0;
        allpos = allpos && posv[c] >= 0;
        alldst = alldst && dstv[c] >= 0;
      }
      // staging buffer free in this chunk: the other chunk parity's (its
      // readers all passed the previous chunk's closing barrier), or the
      // group's own one after its exchange reads
      float* tbuf = G == 1 ? stg + (buf ^ 1) * (128 * 17) : sb;
      bool run = rope && posv[0] >= 0;   // all 16 positions consecutive
#pragma unroll
      for (int c = 1; c < 16; ++c) run = run && posv[c] == posv[0] + c;
      float2 cs = rope ? sh.rope_base[c0 >> 4][fi] : make_float2(1.f, 0.f);
      uint16_t ov[16];
      float xf[16];
      const float sg = lo ? -1.f : 1.f;   // rotate-half sign of this row
      if (run) {
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          xf[c] = fmaf(sg * other[c], cs.y, v[c] * cs.x);
          cs = make_float2(cs.x * rot.x - cs.y * rot.y, cs.y * rot.x + cs.x * rot.y);
        }
      } else {
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          float x = v[c];
          if (rope) {
            const int pos = posv[c];
            const float2 t = pos >= 0 ? e.rope[static_cast<size_t>(pos) * half + fi] : make_float2(1.f, 0.f);
            x = fmaf(sg * other[c], t.y, x * t.x);
          }
          xf[c] = x;
        }
      }
      if (kind == EPI_QKV_ROPE && e.qkv_f16) {
#pragma unroll
        for (int c = 0; c < 16; ++c) ov[c] = f32_to_f16(xf[c]);
      } else {
#pragma unroll
        for (int c = 0; c < 16; ++c) ov[c] = f32_to_bf16(xf[c]);
      }
      if (kind == EPI_KV_APPEND && e.kv_q8) {
        // 8-bit pages: the 32 lanes of this warp are 32 consecutive values of
        // one head row (tile rows 32q .. 32q+31 of a K or V region), i.e. one
        // block per token (column). Scale d = max|x| / 127, codes round(x / d)
        // halves away from zero (stored as the byte code + 128), d stored as
        // fp16 by lane c for column c.
        const int layer = e.layer0 + (reg >> 1), blk = di >> 5, nb = d >> 5;
        const bool is_v = (reg & 1) != 0;
        const size_t hb = q8_head_bytes(d);
        uint8_t* pb = reinterpret_cast<uint8_t*>(e.pool);
        float amax[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) amax[c] = fabsf(xf[c]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
          for (int c = 0; c < 16; ++c) amax[c] = fmaxf(amax[c], __shfl_xor_sync(0xffffffffu, amax[c], o));
        }
        uint32_t qb[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const float dd = amax[c] / 127.f;
          float t = dd > 0.f ? xf[c] / dd : 0.f;
          t = fminf(fmaxf(truncf(t + copysignf(0.5f, t)), -127.f), 127.f);
          qb[c] = static_cast<uint32_t>(static_cast<int>(t) + 128);   // stored offset-binary: code + 128
        }
        auto region = [&](int dst) {   // byte offset of this head's region of the token's page
          const int page = dst / (2 * e.n_kv_heads * kPage);
          return ((static_cast<size_t>(layer) * e.pool_pages + page) * e.n_kv_heads + hd) * hb;
        };
        // the chunk's 16 tokens at consecutive slots of one page
        bool qrun = dstv[0] >= 0 && (dstv[0] & (kPage - 1)) + 16 <= kPage;
#pragma unroll
        for (int c = 1; c < 16; ++c) qrun = qrun && dstv[c] == dstv[0] + c;
        if (is_v && qrun) {   // one row of the transposed code tile: 16 contiguous bytes
          const int slot0 = dstv[0] & (kPage - 1);
          uint8_t* p = pb + region(dstv[0]) + q8_vcode_off(d) + static_cast<size_t>(di) * kPage + slot0;
          uint32_t w[4];
#pragma unroll
          for (int k = 0; k < 4; ++k)
            w[k] = qb[4 * k] | (qb[4 * k + 1] << 8) | (qb[4 * k + 2] << 16) | (qb[4 * k + 3] << 24);
          if ((slot0 & 15) == 0) {
            *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
          } else if ((slot0 & 3) == 0) {
#pragma unroll
            for (int k = 0; k < 4; ++k) reinterpret_cast<uint32_t*>(p)[k] = w[k];
          } else {
#pragma unroll
            for (int c = 0; c < 16; ++c) p[c] = static_cast<uint8_t>(qb[c]);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const int dst = dstv[c];
            if (dst < 0) continue;
            const int slot = dst & (kPage - 1);
            pb[region(dst) + (is_v ? q8_vcode_off(d) + static_cast<size_t>(di) * kPage + slot
                                   : static_cast<size_t>(slot) * d + di)] = static_cast<uint8_t>(qb[c]);
          }
        }
        // lane c stores column c's scale
        float my_amax = 0.f;
        int my_dst = -1;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          if (lane == c) {
            my_amax = amax[c];
            my_dst = dstv[c];
          }
        }
        if (lane < 16 && my_dst >= 0) {
          const int slot = my_dst & (kPage - 1);
          const size_t so = is_v ? q8_vscale_off(d) + (static_cast<size_t>(blk) * kPage + slot) * 2
                                 : q8_kscale_off(d) + (static_cast<size_t>(slot) * nb + blk) * 2;
          *reinterpret_cast<__half*>(pb + region(my_dst) + so) = __float2half_rn(my_amax / 127.f);
        }
      } else {
      // KV append, value rows: the chunk's 16 tokens at consecutive slots of
      // one page are 32 contiguous bytes of this row of the transposed value
      // tile, written with the widest aligned stores (the per-token path
      // would make 16 two-byte stores to 16 sectors shared with no other lane)
      bool vrun = kind == EPI_KV_APPEND && (reg & 1) && dstv[0] >= 0 && (dstv[0] & (kPage - 1)) + 16 <= kPage;
#pragma unroll
      for (int c = 1; c < 16; ++c) vrun = vrun && dstv[c] == dstv[0] + c;
      if (vrun) {
        const int slot0 = dstv[0] & (kPage - 1);
        const int layer = e.layer0 + (reg >> 1);
        uint16_t* p = e.pool +
                      (static_cast<size_t>(layer) * e.pool_pages * 2 * e.n_kv_heads * kPage +
                       static_cast<size_t>(dstv[0] - slot0)) * d +
                      static_cast<size_t>(e.n_kv_heads) * kPage * d + (static_cast<size_t>(hd) * d + di) * kPage + slot0;
        uint32_t w[8];
        if ((slot0 & 1) == 0) {
#pragma unroll
          for (int c = 0; c < 8; ++c)
            w[c] = static_cast<uint32_t>(ov[2 * c]) | (static_cast<uint32_t>(ov[2 * c + 1]) << 16);
          if ((slot0 & 7) == 0) {
            uint4* q4 = reinterpret_cast<uint4*>(p);
            q4[0] = make_uint4(w[0], w[1], w[2], w[3]);
            q4[1] = make_uint4(w[4], w[5], w[6], w[7]);
          } else {
            uint32_t* q2 = reinterpret_cast<uint32_t*>(p);
#pragma unroll
            for (int c = 0; c < 8; ++c) q2[c] = w[c];
          }
        } else {   // odd first slot: one value, seven aligned pairs, one value
          p[0] = ov[0];
          uint32_t* q2 = reinterpret_cast<uint32_t*>(p + 1);
#pragma unroll
          for (int c = 0; c < 7; ++c)
            q2[c] = static_cast<uint32_t>(ov[2 * c + 1]) | (static_cast<uint32_t>(ov[2 * c + 2]) << 16);
          p[15] = ov[15];
        }
      } else if (kind == EPI_QKV_ROPE && reg != 2 && allpos && m0 + c0 + 16 <= a.M) {   // whole chunk of q or k
        const size_t ld = static_cast<size_t>(reg == 0 ? e.n_q_heads : e.n_kv_heads) * d;
        uint16_t* p0 = (reg == 0 ? e.out_q : e.out_k) + static_cast<size_t>(m0 + c0) * ld + (rf - f);
        store_chunk_transposed(ov, r, tbuf, grp, [&](int c, int seg) { return p0 + static_cast<size_t>(c) * ld + seg; });
      } else if (kind == EPI_KV_APPEND && !(reg & 1) && alldst) {   // keys of 16 tokens: [slot][d] rows of pages
        const int layer = e.layer0 + (reg >> 1), rf0 = rf - f;
        store_chunk_transposed(ov, r, tbuf, grp, [&](int c, int seg) -> uint16_t* {
          const int dst = sh.row_dst[c0 + c], slot = dst & (kPage - 1);
          const int hk = (rf0 + seg) / d, dk = rf0 + seg - hk * d;
          const size_t lp = (static_cast<size_t>(layer) * e.pool_pages * 2 * e.n_kv_heads * kPage +
                             static_cast<size_t>(dst - slot)) * d;
          return e.pool + lp + (static_cast<size_t>(hk) * kPage + slot) * d + dk;
        });
      } else
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const int m = m0 + c0 + c;
        if (m >= a.M || posv[c] < 0) continue;
        if (kind == EPI_QKV_ROPE) {
          if (reg == 2) {   // values transposed per (sequence, head): [d][64 slots]
            const int i = m / e.meta.B, j = m - i * e.meta.B;
            e.out_v[((static_cast<size_t>(i) * e.n_kv_heads + hd) * d + di) * kPage + j] = ov[c];
          } else {
            uint16_t* base = reg == 0 ? e.out_q : e.out_k;
            const size_t ld = static_cast<size_t>(reg == 0 ? e.n_q_heads : e.n_kv_heads) * d;
            base[static_cast<size_t>(m) * ld + rf] = ov[c];
          }
        } else {
          const int dst = dstv[c];
          if (dst < 0) continue;
          const int layer = e.layer0 + (reg >> 1), slot = dst & (kPage - 1);
          // elements of (layer, page): keys [n_kv][64][d], then values [n_kv][d][64]
          const size_t lp = (static_cast<size_t>(layer) * e.pool_pages * 2 * e.n_kv_heads * kPage +
                             static_cast<size_t>(dst - slot)) * d;
          const size_t off = (reg & 1) ? static_cast<size_t>(e.n_kv_heads) * kPage * d +
                                             (static_cast<size_t>(hd) * d + di) * kPage + slot
                                       : (static_cast<size_t>(hd) * kPage + slot) * d + di;
          e.pool[lp + off] = ov[c];
        }
      }
      }
    }
#pragma unroll
    for (int c = 0; c < 16; ++c) {
#pragma unroll
      for (int k = 0; k < kAhead; ++k) pc0[k][c] = pn0[k][c];
      ra[c] = rb[c];
      rb[c] = rc[c];
    }
  }
  epi_bar(grp);
}


template <int BN, int EC>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ AMaps amaps, const __grid_constant__ CUtensorMap xmap,
                const __grid_constant__ GemmArgs a, const __grid_constant__ ARegions rg,
                const __grid_constant__ GemmEpi e) {
  using C = Cfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* stg = reinterpret_cast<float*>(smem + C::kStages * C::kStageBytes);
  __shared__ __align__(8) uint64_t full[C::kStages];
  __shared__ __align__(8) uint64_t empty[C::kStages];
  __shared__ __align__(8) uint64_t acc_full[2];
  __shared__ __align__(8) uint64_t acc_empty[2];
  __shared__ __align__(8) uint64_t pair_rdy;   // cluster peer's ring is idle (count 1)
  __shared__ __align__(8) uint64_t pair_dat;   // cluster peer's half sums have landed here (count 128)
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;
  __shared__ EpiShared esh;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = blockIdx.x;
  const long long u0 = unit_begin(g, a), u1 = unit_begin(g + 1, a);
  const int n_units = static_cast<int>(u1 - u0);
  const int kb = a.k_blocks;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);
    }
    mbar_init(&pair_rdy, 1);
    mbar_init(&pair_dat, 128);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&xmap);
    for (int i = 0; i < rg.n_regions && i < kMaxAMaps; ++i) tma_prefetch_desc(&amaps.m[i]);
  }
  if (warp == 1) tmem_alloc(&tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // the cluster peer arrives on this CTA's barriers only after they exist
  if (a.csplit) cluster_sync_all();
  const uint32_t tmem = tmem_slot;
  grid_dep_launch();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      // Walks its (tile, k-block) units incrementally: the weight rows and
      // token rows are recomputed only when the tile changes.
      const uint64_t wpol = policy_evict_first();
      struct Cursor {
        int t, k, ml, rl, mh, rh, brow;
      };
      auto at_tile = [&](Cursor& c) {
        const int tn = c.t / a.m_tiles;
        weight_rows(rg, tn, c.ml, c.rl, c.mh, c.rh);
        c.brow = (c.t - tn * a.m_tiles) * BN;
      };
      auto advance = [&](Cursor& c) {
        if (++c.k == kb) {
          c.k = 0;
          ++c.t;
          at_tile(c);
        }
      };
      Cursor ca;
      ca.t = static_cast<int>(u0 / kb);
      ca.k = static_cast<int>(u0 - static_cast<long long>(ca.t) * kb);
      at_tile(ca);
      Cursor cb = ca;
      auto load_a = [&](int i, const Cursor& c) {
        uint8_t* sa = smem + (i % C::kStages) * C::kStageBytes;
        tma_load_2d_hint(sa, &amaps.m[c.ml], &full[i % C::kStages], c.k * kTileK, c.rl, wpol);
        tma_load_2d_hint(sa + kABytes / 2, &amaps.m[c.mh], &full[i % C::kStages], c.k * kTileK, c.rh, wpol);
      };
      auto load_b = [&](int i, const Cursor& c) {
        uint8_t* sb = smem + (i % C::kStages) * C::kStageBytes + kABytes;
        tma_load_2d(sb, &xmap, &full[i % C::kStages], c.k * kTileK, c.brow);
      };
      // Weights do not depend on the previous kernel: start streaming them
      // before waiting for it (programmatic dependent launch).
      const int pre = min(n_units, C::kStages);
      for (int i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(&full[i], C::kStageBytes);
        load_a(i, ca);
        advance(ca);
      }
      grid_dep_wait();
      for (int i = 0; i < pre; ++i) {
        load_b(i, cb);
        advance(cb);
      }
      int issued = pre;
      for (int i = pre; i < n_units; ++i) {
        const int s = i % C::kStages;
        if (!mbar_wait(&empty[s], ((i / C::kStages) & 1) ^ 1, &abort_flag)) {
          abort_flag = 1;
          latch_status(a.status, kDevTimeout);
          break;
        }
        mbar_arrive_expect_tx(&full[s], C::kStageBytes);
        load_a(i, ca);
        load_b(i, ca);
        advance(ca);
        ++issued;
      }
      if (abort_flag) {  // drain copies still in flight before shared memory is released
        for (int i = max(0, issued - C::kStages); i < issued; ++i)
          mbar_wait(&full[i % C::kStages], (i / C::kStages) & 1);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      constexpr uint32_t idesc = idesc_bf16_f32(kTileN, BN);
      grid_dep_wait();
      int i = 0, seg = 0;
      for (long long u = u0; u < u1 && !abort_flag; ++seg) {
        const long long t = u / kb;
        const long long seg_end = min(u1, (t + 1) * kb);
        const int buf = seg & 1;
        if (!mbar_wait(&acc_empty[buf], ((seg >> 1) & 1) ^ 1, &abort_flag)) {
          abort_flag = 1;
          latch_status(a.status, kDevTimeout);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + buf * BN;
        for (long long v = u; v < seg_end; ++v, ++i) {
          const int s = i % C::kStages;
          if (!mbar_wait(&full[s], (i / C::kStages) & 1, &abort_flag)) {
            abort_flag = 1;
            latch_status(a.status, kDevTimeout);
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + s * C::kStageBytes);
          const uint64_t ad = sdesc_kmajor_sw128(sa);
          const uint64_t bd = sdesc_kmajor_sw128(sa + kABytes);
#pragma unroll
          for (int k = 0; k < kTileK / 16; ++k)
            tc_mma_bf16(d_tmem, ad + 2 * k, bd + 2 * k, idesc, (v != u || k != 0) ? 1u : 0u);
          tc_commit(&empty[s]);
        }
        tc_commit(&acc_full[buf]);
        u = seg_end;
      }
    }
  } else {
    // ---------------- epilogue warps ----------------
    grid_dep_wait();
    const int q = warp & 3;                 // TMEM lane quarter of this warp
    const int r = q * 32 + lane;            // TMEM lane = tile row slot
    const uint32_t trow = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const size_t slot_elems = static_cast<size_t>(kTileN) * BN;
    int seg = 0;
    for (long long u = u0; u < u1; ++seg) {
      const int t = static_cast<int>(u / kb);
      const long long seg_end = min(u1, static_cast<long long>(t + 1) * kb);
      const bool whole = (u == static_cast<long long>(t) * kb) && (seg_end == static_cast<long long>(t + 1) * kb);
      const int buf = seg & 1;
      // Column constants (RMSNorm scales, positions, RoPE bases) and a
      // one-chunk tile's residual input do not depend on the accumulator:
      // they are fetched while the MMAs run, whether or not this CTA ends up
      // finishing the tile.
      const int tn0 = t / a.m_tiles, m0 = (t - tn0 * a.m_tiles) * BN;
      // columns (tokens) this CTA finishes: all, or its half of a cluster-split tile
      const int cbeg = a.csplit ? (g & 1) * (BN / 2) : 0;
      const int cend = a.csplit ? cbeg + BN / 2 : BN;
      tile_cols_prepare<BN, EC>(a, e, m0, r, esh);
      const EpiPre pp = epi_pre<EC>(a, rg, e, t, r);
      float rpre[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) rpre[c] = 0.f;
      // A CTA that owns exactly one whole tile leaves the other accumulator
      // buffer unused: the residual add's input tile is loaded into it while
      // the MMAs run, so the epilogue reads it from TMEM.
      uint32_t pre = 0;
      if constexpr (EC == kEcNorm) {
        if (e.kind == EPI_RESID && (whole || a.csplit) && u0 == u && u1 == seg_end) {
          const int n = tn0 * kTileN + r;
          pre = trow + (buf ^ 1) * BN;
#pragma unroll 1
          for (int c0 = cbeg; c0 < cend; c0 += 32) {
            float xv[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              const int m = m0 + c0 + c;
              xv[c] = (n < a.N && m < a.M) ? __ldcg(e.out_f32 + static_cast<size_t>(m) * e.ld_out + n) : 0.f;
            }
            tmem_store32(pre + c0, xv);
          }
          tmem_wait_st_gk();
        } else if (BN == 16 && e.kind == EPI_RESID) {
          load_resid(a, e, m0, 0, tn0 * kTileN + r, rpre);
        }
      }
      if (!mbar_wait(&acc_full[buf], (seg >> 1) & 1, &abort_flag)) {
        abort_flag = 1;
        latch_status(a.status, kDevTimeout);
      }
      epi_bar();
      if (r == 0) esh.flag[0] = abort_flag;   // one reader, so all epilogue threads agree
      epi_bar();
      if (esh.flag[0]) break;
      tc_fence_after();
      const uint32_t tb = trow + buf * BN;
      bool finish = whole;
      int first = g, last = g;
      const float* speer = nullptr;
      if (a.csplit) {
        // Cluster pair: each CTA sends the peer the half-K sums of the
        // peer's columns, straight into the peer's (idle) operand ring, and
        // finishes its own columns with the peer's sums added.
        const uint32_t peer = static_cast<uint32_t>(g & 1) ^ 1u;
        const int pbeg = static_cast<int>(peer) * (BN / 2);
        // all of this CTA's MMAs have completed, so its ring is idle
        if (r == 0) mbar_arrive_remote(mapa_shared(smem_u32(&pair_rdy), peer));
        bool ok = mbar_wait_cluster(&pair_rdy, 0, &abort_flag);
        if (ok) {
          const uint32_t dst = mapa_shared(smem_u32(smem), peer) + static_cast<uint32_t>(r) * 4u;
#pragma unroll 1
          for (int c0 = 0; c0 < BN / 2; c0 += 16) {
            float v[16];
            tmem_ld16(tb + pbeg + c0, v);
#pragma unroll
            for (int c = 0; c < 16; ++c) st_cluster_f32(dst + static_cast<uint32_t>((c0 + c) * 128) * 4u, v[c]);
          }
          mbar_arrive_remote(mapa_shared(smem_u32(&pair_dat), peer));
          ok = mbar_wait_cluster(&pair_dat, 0, &abort_flag);
        }
        if (!ok) {
          abort_flag = 1;
          latch_status(a.status, kDevTimeout);
        }
        epi_bar();
        if (r == 0) esh.flag[0] = abort_flag;
        epi_bar();
        if (esh.flag[0]) break;
        speer = reinterpret_cast<const float*>(smem);
        finish = true;
      } else if (!whole) {
        // park this segment's partial sum in the CTA's slot, then take a ticket
        const int side = (u == u0) ? 0 : 1;
        park_partial<BN>(tb, part_row(a.partial + (static_cast<size_t>(g) * 2 + side) * slot_elems, r));
        first = cta_of(static_cast<long long>(t) * kb, a);
        last = cta_of(static_cast<long long>(t + 1) * kb - 1, a);
        __threadfence();
        epi_bar();
        if (r == 0) {
          const int tk = atomicAdd(a.tickets + t, 1);
          esh.flag[0] = (tk == last - first);
          if (tk == last - first) a.tickets[t] = 0;
        }
        epi_bar();
        finish = esh.flag[0] != 0;
        if (finish) __threadfence();
      }
      if (finish) {
        epilogue_tile<BN, EC>(a, rg, e, g, t, first, last, tb, r, esh, stg, pre, rpre, pp, cbeg, cend, speer,
                              static_cast<long long>(t) * kb);
        if constexpr (EC == kEcArgmax) argmax_tile_done(a, e, esh, r, (a.csplit ? 2 : 1) * a.n_tiles * a.m_tiles);
      }
      // hand the TMEM buffer back to the MMA warp
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
      u = seg_end;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  // no CTA leaves while its cluster peer may still write into its shared memory
  if (a.csplit) cluster_sync_all();
}

// ---------------------------------------------------------------------------
// CTA-pair GEMM (cta_group::2). A cluster of two CTAs computes a tile of two
// weight tiles (256 rows) by 256 tokens: each CTA stages its own weight tile
// and half of the tokens (128 rows), and one thread of the first CTA issues
// M = 256, N = 256 MMAs that read both CTAs' shared memory. Each CTA's TMEM
// receives its weight tile's rows over all 256 tokens, so the epilogue is the
// single-CTA one. One MMA instruction does twice the work of a single-CTA
// 256-token one at the same issue cost (the issuing thread's fixed cost per
// k-block is what limits single-CTA tensor-bound tiles), and a stage is 32 KB,
// so six fit. Pairs take whole pair tiles round-robin; a pair's second weight
// tile past N (odd tile count) loads zeros and stores nothing.
constexpr int kEpiGroups = 2;                     // epilogue groups of the pair kernel
constexpr int kPairThreads = 64 + kEpiGroups * 128; // TMA warp, MMA warp, epilogue groups
struct PairCfg {
  static constexpr int BN = 256;
  static constexpr int kBHalfBytes = (BN / 2) * kTileK * 2;   // 16 KB
  static constexpr int kStageBytes = kABytes + kBHalfBytes;     // 32 KB per CTA
  static constexpr int kStages = 6;
  static constexpr int kTmemCols = 2 * BN;                      // two accumulators
  static constexpr int kStgBytes = kEpiGroups * 128 * 17 * 4;   // one exchange buffer per epilogue group
  static constexpr int kSmem = kStages * kStageBytes + kStgBytes + 1024;
};

// MODE 1: pairs take whole pair tiles round-robin.
// MODE 2 (KS = 2): a cluster of four CTAs, two pairs over the two halves of
// the k-blocks of one pair tile; the CTAs holding the same weight tile in the
// two pairs exchange the half sums of each other's 128 token columns through
// distributed shared memory (as the single-CTA cluster split does) and each
// finishes its own 128 columns. Used when four CTAs per pair tile fit one
// wave, which single pairs would leave half idle.
// MODE 3: stream-K over pairs. Pair p owns an equal contiguous range of
// (pair tile, k-block) units, so every SM pair has the same MMA work whatever
// the tile count. Each CTA of the pair holds one weight tile's 128 rows of
// the pair tile, an ordinary 128 x 256 tile: a segment that does not cover a
// whole tile is parked in the CTA's partial slot and the tile is finished by
// the last CTA (of those holding the same weight tile) to take its ticket, as
// in the single-CTA kernel.
template <int EC, int MODE>
__global__ void __launch_bounds__(kPairThreads, 1)
    gemm_pair_kernel(const __grid_constant__ AMaps amaps, const __grid_constant__ CUtensorMap xmap,
                     const __grid_constant__ GemmArgs a, const __grid_constant__ ARegions rg,
                     const __grid_constant__ GemmEpi e) {
  using P = PairCfg;
  constexpr int BN = P::BN;
  constexpr int KS = MODE == 2 ? 2 : 1;
  constexpr bool SK = MODE == 3;
  constexpr int CL = 2 * KS;   // CTAs per cluster
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* stg = reinterpret_cast<float*>(smem + P::kStages * P::kStageBytes);
  __shared__ __align__(8) uint64_t full[P::kStages];    // the pair's first CTA's count both CTAs' bytes
  __shared__ __align__(8) uint64_t empty[P::kStages];
  __shared__ __align__(8) uint64_t acc_full[2];
  __shared__ __align__(8) uint64_t acc_empty[2];        // the pair's first CTA's: every epilogue warp of each CTA
  __shared__ __align__(8) uint64_t split_rdy;           // KS = 2: the other pair's CTA's ring is idle (count 1)
  __shared__ __align__(8) uint64_t split_dat;           // KS = 2: its half sums have landed here (count 128)
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;
  __shared__ EpiShared esh;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = blockIdx.x;
  const uint32_t crank = static_cast<uint32_t>(g % CL);   // rank in the cluster
  const uint32_t member = crank & 1u;                      // weight tile of the pair tile this CTA stages
  const uint32_t half = crank >> 1;                        // KS = 2: which half of the k-blocks
  const uint32_t lead = crank & ~1u;                       // the pair's first CTA
  const uint16_t pair_mask = static_cast<uint16_t>(0x3u << lead);
  const int pair = g / CL, n_pairs = static_cast<int>(gridDim.x) / CL;
  const int kb = a.k_blocks;
  const int kbeg = KS == 2 ? static_cast<int>(half) * (kb >> 1) : 0;
  const int kend = KS == 2 && half == 0 ? (kb >> 1) : kb;
  const int nk = kend - kbeg;
  const int pair_tiles = ((a.n_tiles + 1) >> 1) * a.m_tiles;
  // columns (tokens) this CTA finishes
  const int cbeg = KS == 2 ? static_cast<int>(half) * (BN / 2) : 0;
  const int cend = KS == 2 ? cbeg + BN / 2 : BN;
  // MODE 3: this pair's range of (pair tile, k-block) units
  const long long su0 = SK ? unit_begin(pair, a) : 0, su1 = SK ? unit_begin(pair + 1, a) : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < P::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 2 * 4 * kEpiGroups);   // every epilogue warp of both CTAs
    }
    mbar_init(&split_rdy, 1);
    mbar_init(&split_dat, 128 * kEpiGroups);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&xmap);
    for (int i = 0; i < rg.n_regions && i < kMaxAMaps; ++i) tma_prefetch_desc(&amaps.m[i]);
  }
  if (warp == 1) tmem_alloc_pair(&tmem_slot, P::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // the other CTAs signal this CTA's barriers only after they exist
  cluster_sync_all();
  const uint32_t tmem = tmem_slot;
  grid_dep_launch();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (every CTA) ----------------
      const uint64_t wpol = policy_evict_first();
      const uint32_t lead_full = mapa_shared(smem_u32(&full[0]), lead);   // the pair's first CTA's full barriers
      struct Cur {
        int pt, k, ml, rl, mh, rh, brow;
      };
      auto at_tile = [&](Cur& c) {
        const int pr = c.pt / a.m_tiles, tm = c.pt - pr * a.m_tiles;
        weight_rows(rg, 2 * pr + static_cast<int>(member), c.ml, c.rl, c.mh, c.rh);
        c.brow = tm * BN + static_cast<int>(member) * (BN / 2);
      };
      auto advance = [&](Cur& c) {
        if (++c.k == kend) {
          c.k = kbeg;
          c.pt += SK ? 1 : n_pairs;
          if (c.pt < pair_tiles) at_tile(c);
        }
      };
      int n_units;
      Cur ca{pair, kbeg, 0, 0, 0, 0, 0};
      if constexpr (SK) {
        n_units = static_cast<int>(su1 - su0);
        ca.pt = static_cast<int>(su0 / kb);
        ca.k = static_cast<int>(su0 - static_cast<long long>(ca.pt) * kb);
      } else {
        n_units = pair < pair_tiles ? ((pair_tiles - 1 - pair) / n_pairs + 1) * nk : 0;
      }
      if (n_units > 0) at_tile(ca);
      Cur cb = ca;
      auto load_a = [&](int i, const Cur& c) {
        const int s = i % P::kStages;
        if (member == 0) mbar_arrive_expect_tx(&full[s], 2 * P::kStageBytes);
        uint8_t* sa = smem + s * P::kStageBytes;
        tma_load_2d_pair(sa, &amaps.m[c.ml], lead_full + 8u * s, c.k * kTileK, c.rl, wpol);
        tma_load_2d_pair(sa + kABytes / 2, &amaps.m[c.mh], lead_full + 8u * s, c.k * kTileK, c.rh, wpol);
      };
      auto load_b = [&](int i, const Cur& c) {
        const int s = i % P::kStages;
        tma_load_2d_pair_nohint(smem + s * P::kStageBytes + kABytes, &xmap, lead_full + 8u * s, c.k * kTileK,
                                c.brow);
      };
      // weights do not depend on the previous kernel: the first stages' are
      // requested before waiting for it
      const int pre = min(n_units, P::kStages);
      for (int i = 0; i < pre; ++i) {
        load_a(i, ca);
        advance(ca);
      }
      grid_dep_wait();
      for (int i = 0; i < pre; ++i) {
        load_b(i, cb);
        advance(cb);
      }
      for (int i = pre; i < n_units; ++i) {
        const int s = i % P::kStages;
        if (!mbar_wait(&empty[s], ((i / P::kStages) & 1) ^ 1, &abort_flag)) {
          abort_flag = 1;
          latch_status(a.status, kDevTimeout);
          break;
        }
        load_a(i, ca);
        load_b(i, ca);
        advance(ca);
      }
      if (abort_flag) {
        // copies in flight complete on the pair's first CTA's barriers: give
        // them time to land before shared memory is released
        const unsigned long long t0 = global_ns();
        while (global_ns() - t0 < 50000ull) {
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && member == 0) {
      // ---------------- MMA issuer (the pair's first CTA) ----------------
      constexpr uint32_t idesc = idesc_bf16_f32(2 * kTileN, BN);
      grid_dep_wait();
      int i = 0, j = 0;
      // segments: whole pair tiles (MODE 1, 2), or the stretches of this
      // pair's unit range inside one pair tile (MODE 3)
      long long su = su0;
      for (int pt = SK ? 0 : pair; (SK ? su < su1 : pt < pair_tiles) && !abort_flag; pt += n_pairs, ++j) {
        int seg_k = nk;
        if constexpr (SK) {
          const long long tp = su / kb;
          const long long se = min(su1, (tp + 1) * kb);
          seg_k = static_cast<int>(se - su);
          su = se;
        }
        const int buf = j & 1;
        if (!mbar_wait(&acc_empty[buf], ((j >> 1) & 1) ^ 1, &abort_flag)) {
          abort_flag = 1;
          latch_status(a.status, kDevTimeout);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + buf * BN;
        for (int k = 0; k < seg_k; ++k, ++i) {
          const int s = i % P::kStages;
          if (!mbar_wait(&full[s], (i / P::kStages) & 1, &abort_flag)) {
            abort_flag = 1;
            latch_status(a.status, kDevTimeout);
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + s * P::kStageBytes);
          const uint64_t ad = sdesc_kmajor_sw128(sa);
          const uint64_t bd = sdesc_kmajor_sw128(sa + kABytes);
#pragma unroll
          for (int kk = 0; kk < kTileK / 16; ++kk)
            tc_mma_bf16_pair(d_tmem, ad + 2 * kk, bd + 2 * kk, idesc, (k != 0 || kk != 0) ? 1u : 0u);
          tc_commit_pair(&empty[s], pair_mask);
        }
        tc_commit_pair(&acc_full[buf], pair_mask);
      }
    }
  } else {
    // ---------------- epilogue warps (every CTA) ----------------
    // Two groups of four warps (one per TMEM lane quarter); group grp drains
    // columns [gcb, gce), half of this CTA's columns. Decisions every thread
    // must share (give up after a failed wait, finish a tile) are taken once
    // for both groups behind the 256-thread barrier.
    grid_dep_wait();
    const int grp = (warp - 2) >> 2;
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const int et = threadIdx.x - 64;   // epilogue thread 0 .. 255
    const uint32_t trow = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const uint32_t lead_acc_empty = mapa_shared(smem_u32(&acc_empty[0]), lead);
    const size_t slot_elems = static_cast<size_t>(kTileN) * BN;
    const int gw = (cend - cbeg) / kEpiGroups;
    const int gcb = cbeg + grp * gw, gce = gcb + gw;
    float* gstg = stg;   // epilogue_tile picks the group's buffer
    int j = 0;
    long long su = su0;
    for (int pt0 = SK ? 0 : pair; SK ? su < su1 : pt0 < pair_tiles; pt0 += n_pairs, ++j) {
      int pt = pt0;
      long long seg_u = 0, seg_end = 0;
      if constexpr (SK) {
        pt = static_cast<int>(su / kb);
        seg_u = su;
        seg_end = min(su1, static_cast<long long>(pt + 1) * kb);
        su = seg_end;
      }
      const int pr = pt / a.m_tiles, tm = pt - pr * a.m_tiles;
      const int tn = 2 * pr + static_cast<int>(member);
      const int t = tn * a.m_tiles + tm;   // this CTA's tile
      const int buf = j & 1;
      tile_cols_prepare<BN, EC>(a, e, tm * BN, r, esh, gcb, gce, grp);
      const EpiPre pp = epi_pre<EC>(a, rg, e, t, r);
      float rpre[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) rpre[c] = 0.f;
      // KS = 2 (one pair tile per cluster): the residual input of this CTA's
      // columns goes into the spare accumulator while the MMAs run
      uint32_t pre = 0;
      if constexpr (KS == 2 && EC == kEcNorm) {
        if (e.kind == EPI_RESID && tn < a.n_tiles) {
          const int n = tn * kTileN + r, m0 = tm * BN;
          pre = trow + (buf ^ 1) * BN;
#pragma unroll 1
          for (int c0 = gcb; c0 < gce; c0 += 32) {
            float xv[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              const int m = m0 + c0 + c;
              xv[c] = (n < a.N && m < a.M) ? __ldcg(e.out_f32 + static_cast<size_t>(m) * e.ld_out + n) : 0.f;
            }
            tmem_store32(pre + c0, xv);
          }
          tmem_wait_st_gk();
        }
      }
      if (!mbar_wait(&acc_full[buf], (j >> 1) & 1, &abort_flag)) {
        abort_flag = 1;
        latch_status(a.status, kDevTimeout);
      }
      epi_bar_all();
      if (et == 0) esh.flag[0] = abort_flag;
      epi_bar_all();
      if (esh.flag[0]) break;
      tc_fence_after();
      const uint32_t tb = trow + buf * BN;
      const float* speer = nullptr;
      if constexpr (KS == 2) {
        // send the other half's CTA (same weight tile) the sums of its
        // columns, straight into its idle ring, and take the sums of ours;
        // group grp sends its share of them
        const uint32_t other = crank ^ 2u;
        const int obeg = static_cast<int>(half ^ 1u) * (BN / 2) + grp * gw;
        if (et == 0) mbar_arrive_remote(mapa_shared(smem_u32(&split_rdy), other));
        bool ok = mbar_wait_cluster(&split_rdy, 0, &abort_flag);
        if (ok) {
          const uint32_t dst = mapa_shared(smem_u32(smem), other) + static_cast<uint32_t>(grp * gw * 128 + r) * 4u;
#pragma unroll 1
          for (int c0 = 0; c0 < gw; c0 += 16) {
            float v[16];
            tmem_ld16(tb + obeg + c0, v);
#pragma unroll
            for (int c = 0; c < 16; ++c) st_cluster_f32(dst + static_cast<uint32_t>((c0 + c) * 128) * 4u, v[c]);
          }
          mbar_arrive_remote(mapa_shared(smem_u32(&split_dat), other));
          ok = mbar_wait_cluster(&split_dat, 0, &abort_flag);
        }
        if (!ok) {
          abort_flag = 1;
          latch_status(a.status, kDevTimeout);
        }
        epi_bar_all();
        if (et == 0) esh.flag[0] = abort_flag;
        epi_bar_all();
        if (esh.flag[0]) break;
        speer = reinterpret_cast<const float*>(smem) + (gcb - cbeg) * 128;
      }
      if constexpr (SK) {
        // a pair's second weight tile past N (odd tile count) has no rows: no
        // partial, no ticket, nothing to finish
        bool finish = false;
        int first = pair, last = pair;
        const long long tu0 = static_cast<long long>(pt) * kb;
        if (tn < a.n_tiles) {
          finish = seg_u == tu0 && seg_end == tu0 + kb;
          if (!finish) {
            // park this segment's partial sum in the CTA's slot, then take a ticket
            const int side = (seg_u == su0) ? 0 : 1;
            park_partial<BN>(tb, part_row(a.partial + (static_cast<size_t>(g) * 2 + side) * slot_elems, r), gcb, gce);
            first = cta_of(tu0, a);
            last = cta_of(tu0 + kb - 1, a);
            __threadfence();
            epi_bar_all();
            if (et == 0) {
              const int tk = atomicAdd(a.tickets + t, 1);
              esh.flag[0] = (tk == last - first);
              if (tk == last - first) a.tickets[t] = 0;
            }
            epi_bar_all();
            finish = esh.flag[0] != 0;
            if (finish) __threadfence();
          }
        }
        if (finish) {
          epilogue_tile<BN, EC, kEpiGroups>(a, rg, e, pair, t, first, last, tb, r, esh, gstg, 0u, rpre, pp, gcb, gce,
                                            nullptr, tu0, 2, static_cast<int>(member), grp);
          if constexpr (EC == kEcArgmax) argmax_tile_done(a, e, esh, r, kEpiGroups * a.n_tiles * a.m_tiles, grp);
        }
      } else {
        // a pair's second weight tile past N (odd tile count) has no rows to store
        if (tn < a.n_tiles)
          epilogue_tile<BN, EC, kEpiGroups>(a, rg, e, g, t, g, g, tb, r, esh, gstg, pre, rpre, pp, gcb, gce, speer,
                                            static_cast<long long>(t) * kb, 1, 0, grp);
        if constexpr (EC == kEcArgmax) argmax_tile_done(a, e, esh, r, kEpiGroups * KS * 2 * pair_tiles, grp);
      }
      // hand the accumulator back to the pair's first CTA's MMA thread
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(lead_acc_empty + 8u * buf);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, P::kTmemCols);
  }
  // no CTA leaves while another may still read or signal its shared memory
  cluster_sync_all();
}

template <int EC, int MODE>
cudaError_t launch_pair_mode(const AMaps& amaps, const ARegions& rg, const CUtensorMap& xmap, const GemmArgs& a,
                             const GemmEpi& e, cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t err = cudaFuncSetAttribute(gemm_pair_kernel<EC, MODE>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, PairCfg::kSmem);
    if (err != cudaSuccess) return err;
    attr_set = true;
  }
  return launch_pdl_cluster(gemm_pair_kernel<EC, MODE>, dim3(a.grid), dim3(kPairThreads), PairCfg::kSmem,
                            MODE == 2 ? 4 : 2, stream, amaps, xmap, a, rg, e);
}

template <int EC>
cudaError_t launch_pair(const AMaps& amaps, const ARegions& rg, const CUtensorMap& xmap, const GemmArgs& a,
                        const GemmEpi& e, cudaStream_t stream) {
  if (a.pair == 2) return launch_pair_mode<EC, 2>(amaps, rg, xmap, a, e, stream);
  if (a.pair == 3) return launch_pair_mode<EC, 3>(amaps, rg, xmap, a, e, stream);
  return launch_pair_mode<EC, 1>(amaps, rg, xmap, a, e, stream);
}

template <int BN, int EC>
cudaError_t launch_bn(const AMaps& amaps, const ARegions& rg, const CUtensorMap& xmap, const GemmArgs& a,
                      const GemmEpi& e, cudaStream_t stream) {
  using C = Cfg<BN>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t err = cudaFuncSetAttribute(gemm_kernel<BN, EC>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (err != cudaSuccess) return err;
    attr_set = true;
  }
  if (a.csplit)
    return launch_pdl_cluster(gemm_kernel<BN, EC>, dim3(a.grid), dim3(kThreads), C::kSmem, 2, stream, amaps, xmap, a,
                              rg, e);
  return launch_pdl(gemm_kernel<BN, EC>, dim3(a.grid), dim3(kThreads), C::kSmem, stream, amaps, xmap, a, rg, e);
}

template <int EC>
cudaError_t launch_class_bn(const AMaps& amaps, const ARegions& rg, const CUtensorMap& xmap, const GemmArgs& a,
                            const GemmEpi& e, int BN, cudaStream_t stream) {
  if (a.pair) return launch_pair<EC>(amaps, rg, xmap, a, e, stream);
  switch (BN) {
    case 16: return launch_bn<16, EC>(amaps, rg, xmap, a, e, stream);
    case 32: return launch_bn<32, EC>(amaps, rg, xmap, a, e, stream);
    case 64: return launch_bn<64, EC>(amaps, rg, xmap, a, e, stream);
    case 128: return launch_bn<128, EC>(amaps, rg, xmap, a, e, stream);
    default: return launch_bn<256, EC>(amaps, rg, xmap, a, e, stream);
  }
}

// One translation unit per class (gemm_ec_*.cu) defines its launcher.
cudaError_t launch_ec_f32(const AMaps&, const ARegions&, const CUtensorMap&, const GemmArgs&, const GemmEpi&, int,
                          cudaStream_t);
cudaError_t launch_ec_norm(const AMaps&, const ARegions&, const CUtensorMap&, const GemmArgs&, const GemmEpi&, int,
                           cudaStream_t);
cudaError_t launch_ec_rope(const AMaps&, const ARegions&, const CUtensorMap&, const GemmArgs&, const GemmEpi&, int,
                           cudaStream_t);
cudaError_t launch_ec_swiglu(const AMaps&, const ARegions&, const CUtensorMap&, const GemmArgs&, const GemmEpi&, int,
                             cudaStream_t);
cudaError_t launch_ec_argmax(const AMaps&, const ARegions&, const CUtensorMap&, const GemmArgs&, const GemmEpi&, int,
                             cudaStream_t);

}  // namespace gk
}  // namespace dfl
