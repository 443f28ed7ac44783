// gemm_tc.cu - the drafter's dense contractions on the 5th-generation tensor
// cores (tcgen05.mma, fp32 accumulators in TMEM, operands staged by TMA).
//
// Every projection of the drafter pass is OUT^T[N, M] = W[N, K] * X[M, K]^T:
// the weight rows are the UMMA "A" operand (M_mma = 128 rows per tile) and
// the tokens the "B" operand (N_mma = BN, 16..256), so a batch-1 block of 16
// tokens still fills the 128-row tensor-core tile and the kernel streams
// weights at HBM speed; with 512 tokens the same kernel is compute bound.
//
// CTA = 6 warps: warp 0 issues TMA loads into a STAGES-deep ring of shared
// memory stages, warp 1 owns TMEM and issues the MMAs (one elected thread),
// warps 2-5 drain the accumulator (tcgen05.ld) and run the fused epilogue:
//   EPI_F32_STORE  plain fp32 output (fusion projection W_c, tests)
//   EPI_F32_ADD    residual add (attention output and FFN down projections)
//   EPI_QKV_ROPE   q/k/v split with rotate-half RoPE on q and k
//   EPI_SWIGLU     SiLU(gate) * up from paired gate/up weight rows
//   EPI_KV_APPEND  KV injection: RoPE(W_K H_t), W_V H_t scattered to pages
//   EPI_ARGMAX     LM head with the per-row argmax fused; logits never stored
// Split-K: each split writes an fp32 partial; the last CTA of a tile (atomic
// ticket, no spinning) sums them and runs the epilogue.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace dfl {
namespace {

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
  static constexpr int kStgBytes = 128 * 17 * 4;                    // epilogue staging
  static constexpr int kSmem = kStages * kStageBytes + kStgBytes + 1024;
};

struct GemmArgs {
  int M, N, K;
  int k_blocks, n_tiles, m_tiles;
  long long units;     // tiles * k_blocks
  int grid;            // CTAs (stream-K workers)
  float* partial;      // [grid][2][128 * BN] partial tiles
  int* tickets;        // [tiles], zero between launches
  int* status;
};

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

struct EpiShared {
  unsigned long long cand[4][16];
  int row_pos[256];     // QKV_ROPE / KV_APPEND: absolute position of each tile row
  int row_dst[256];     // KV_APPEND: pool row index of (page, slot) without layer/kv/head
  float row_scale[256]; // folded RMSNorm scale of each tile row
  float red[4][16];     // per-warp column sums of squares
  int flag;
};

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

// Per-row metadata of one output tile (rows m0 .. m0+BN-1), computed once by
// all 128 epilogue threads before the tile's chunks are processed.
template <int BN>
__device__ __forceinline__ void tile_rows_prepare(const GemmArgs& a, const GemmEpi& e, int m0, int r, EpiShared& sh) {
  const int kind = e.kind;
  for (int row = r; row < BN; row += 128) {
    const int m = m0 + row;
    float sc = 0.f;
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
    sh.row_scale[row] = sc;
    sh.row_pos[row] = pos;
    sh.row_dst[row] = dst;
  }
  epi_bar();
}


__device__ __forceinline__ int region_of(const ARegions& rg, int tile) {
  int r = 0;
  while (r + 1 < rg.n_regions && tile >= rg.tile_begin[r + 1]) ++r;
  return r;
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

// Final values of one 16-column chunk: v[c] for output feature (tile row) r
// and token m0 + c0 + c. Staging area `stg` holds 128 x 17 floats.
template <int BN>
__device__ __forceinline__ void epilogue_chunk(const GemmArgs& a, const ARegions& rg, const GemmEpi& e, int tile_n,
                                               int m0, int c0, int r, float (&v)[16], float* stg, EpiShared& sh) {
  const int q = r >> 5;
  const int lane = r & 31;
  const int kind = e.kind;
  if (e.in_ss && kind != EPI_ARGMAX) {
    // folded RMSNorm of the input rows: scale each token column
#pragma unroll
    for (int c = 0; c < 16; ++c) v[c] *= sh.row_scale[c0 + c];
  }
  if (kind == EPI_RESID || kind == EPI_NORMSRC) {
    const int n = tile_n * kTileN + r;
    const bool nv = n < a.N;
    const float g = nv ? bf16_to_f32(e.gain[n]) : 0.f;
    float xo[16];
    if (kind == EPI_RESID) {   // all residual loads in flight at once
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const int m = m0 + c0 + c;
        xo[c] = (nv && m < a.M) ? e.out_f32[static_cast<size_t>(m) * e.ld_out + n] : 0.f;
      }
    }
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const int m = m0 + c0 + c;
      float xn = 0.f;
      if (nv && m < a.M) {
        const size_t off = static_cast<size_t>(m) * e.ld_out + n;
        xn = v[c];
        if (kind == EPI_RESID) {
          xn += xo[c];
          e.out_f32[off] = xn;
        }
        e.out_hg[off] = f32_to_bf16(xn * g);
      }
      float sq = xn * xn;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
      if (lane == 0) sh.red[q][c] = sq;
    }
    epi_bar();
    if (r < 16) {
      const int m = m0 + c0 + r;
      if (m < a.M)
        e.out_ss[static_cast<size_t>(tile_n) * e.out_ss_ld + m] = sh.red[0][r] + sh.red[1][r] + sh.red[2][r] + sh.red[3][r];
    }
    epi_bar();
    return;
  }
  if (kind == EPI_F32_STORE || kind == EPI_F32_ADD) {
    const int n = tile_n * kTileN + r;
    if (n < a.N) {
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const int m = m0 + c0 + c;
        if (m < a.M) {
          float* p = e.out_f32 + static_cast<size_t>(m) * e.ld_out + n;
          if (kind == EPI_F32_ADD) *p += v[c]; else *p = v[c];
        }
      }
    }
    return;
  }
  if (kind == EPI_ARGMAX) {
    const int n = tile_n * kTileN + r;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const int m = m0 + c0 + c;
      const bool ok = (n < a.N) && (m < a.M) && !(e.argmax_skip_B > 0 && m % e.argmax_skip_B == 0);
      const uint32_t key = ok ? ordered_key(v[c]) : 0u;
      const uint32_t mx = __reduce_max_sync(0xffffffffu, key);
      const uint32_t hit = __ballot_sync(0xffffffffu, ok && key == mx);
      if (lane == 0) {
        unsigned long long cand = 0ull;
        if (hit) {
          const uint32_t idx = static_cast<uint32_t>(tile_n * kTileN + q * 32 + (__ffs(hit) - 1));
          cand = (static_cast<unsigned long long>(mx) << 32) | (0xFFFFFFFFu - idx);
        }
        sh.cand[q][c] = cand;
      }
    }
    epi_bar();
    if (r < 16) {
      unsigned long long best = sh.cand[0][r];
#pragma unroll
      for (int w = 1; w < 4; ++w) best = sh.cand[w][r] > best ? sh.cand[w][r] : best;
      const int m = m0 + c0 + r;
      if (m < a.M && best) atomicMax(e.keys + m, best);
    }
    epi_bar();
    return;
  }

  // Remaining kinds pair rows of the tile: stage it in shared memory.
#pragma unroll
  for (int c = 0; c < 16; ++c) stg[r * 17 + c] = v[c];
  epi_bar();

  if (kind == EPI_SWIGLU) {
    const int rr = r & 63;
    const int f = tile_n * 64 + rr;
    if (f < e.n_valid) {
      for (int c = r >> 6; c < 16; c += 2) {
        const int m = m0 + c0 + c;
        if (m < a.M) {
          const float g = stg[rr * 17 + c];
          const float u = stg[(rr + 64) * 17 + c];
          e.out_act[static_cast<size_t>(m) * e.n_valid + f] = f32_to_bf16(silu_f(g) * u);
        }
      }
    }
  } else {
    // QKV_ROPE or KV_APPEND
    const int reg = region_of(rg, tile_n);
    const int f = (tile_n - rg.tile_begin[reg]) * kTileN + r;   // feature within the region's matrix
    const int d = e.head_dim, half = d >> 1;
    const int head = f / d, i = f - head * d;
    bool rope;
    uint16_t* base;
    size_t ld;
    int layer = 0, kv = 0;
    if (kind == EPI_QKV_ROPE) {
      rope = reg < 2;
      base = reg == 0 ? e.out_q : (reg == 1 ? e.out_k : e.out_v);
      ld = static_cast<size_t>(reg == 0 ? e.n_q_heads : e.n_kv_heads) * d;
    } else {
      layer = e.layer0 + (reg >> 1);
      kv = reg & 1;
      rope = kv == 0;
      base = e.pool;
      ld = 0;
    }
    const int partner = i < half ? r + half : r - half;
    const int fi = i < half ? i : i - half;
#pragma unroll 4
    for (int c = 0; c < 16; ++c) {
      const int m = m0 + c0 + c;
      const int pos = sh.row_pos[c0 + c];
      if (m >= a.M || pos < 0) continue;
      float x = stg[r * 17 + c];
      if (rope) {
        const float2 cs = e.rope[static_cast<size_t>(pos) * half + fi];
        const float p = stg[partner * 17 + c];
        x = i < half ? (x * cs.x - p * cs.y) : (x * cs.x + p * cs.y);
      }
      if (kind == EPI_QKV_ROPE) {
        base[static_cast<size_t>(m) * ld + f] = f32_to_bf16(x);
      } else {
        const int dst = sh.row_dst[c0 + c];
        if (dst < 0) continue;
        // pool row = ((layer*P + page)*2 + kv)*n_kv + head)*64 + slot
        const size_t row = static_cast<size_t>(layer) * e.pool_pages * 2 * e.n_kv_heads * kPage +
                           static_cast<size_t>(dst) + static_cast<size_t>(kv * e.n_kv_heads + head) * kPage;
        base[row * d + i] = f32_to_bf16(x);
      }
    }
  }
  epi_bar();
}

// Stream-K partition: CTA g owns the contiguous range of (tile, k-block)
// units [unit_begin(g), unit_begin(g + 1)); tiles are ordered so that the m
// tiles of one weight tile are consecutive (weights reused from L2).
__device__ __forceinline__ long long unit_begin(int g, const GemmArgs& a) {
  return static_cast<long long>(g) * a.units / a.grid;
}
__device__ __forceinline__ int cta_of(long long u, const GemmArgs& a) {
  long long g = u * a.grid / a.units;
  while (g + 1 < a.grid && unit_begin(static_cast<int>(g + 1), a) <= u) ++g;
  while (g > 0 && unit_begin(static_cast<int>(g), a) > u) --g;
  return static_cast<int>(g);
}

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

// Persistent, stream-K tcgen05 GEMM. One CTA per SM; each streams its unit
// range through a STAGES-deep TMA ring. Warp 1 accumulates each tile segment
// in one of two TMEM buffers while warps 2-5 drain the other: a segment that
// covers a whole tile goes straight to the epilogue; a partial segment is
// written to the CTA's partial slot and the last CTA to finish a tile (atomic
// ticket) adds the other slots to its own accumulator and runs the epilogue.
template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ AMaps amaps, const __grid_constant__ CUtensorMap xmap,
                const __grid_constant__ GemmArgs a, const __grid_constant__ ARegions rg,
                const __grid_constant__ GemmEpi e) {
  using C = Cfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* stg = reinterpret_cast<float*>(smem + C::kStages * C::kStageBytes);   // 128 x 17 floats
  __shared__ __align__(8) uint64_t full[C::kStages];
  __shared__ __align__(8) uint64_t empty[C::kStages];
  __shared__ __align__(8) uint64_t acc_full[2];
  __shared__ __align__(8) uint64_t acc_empty[2];
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
    const int r = q * 32 + lane;            // tile row = output feature
    const uint32_t trow = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const size_t slot_elems = static_cast<size_t>(kTileN) * BN;
    int seg = 0;
    for (long long u = u0; u < u1; ++seg) {
      const int t = static_cast<int>(u / kb);
      const long long seg_end = min(u1, static_cast<long long>(t + 1) * kb);
      const bool whole = (u == static_cast<long long>(t) * kb) && (seg_end == static_cast<long long>(t + 1) * kb);
      const int buf = seg & 1;
      const int tn = t / a.m_tiles, tm = t - tn * a.m_tiles;
      const int m0 = tm * BN;
      if (!mbar_wait(&acc_full[buf], (seg >> 1) & 1, &abort_flag)) {
        abort_flag = 1;
        latch_status(a.status, kDevTimeout);
      }
      epi_bar();
      if (r == 0) esh.flag = abort_flag;   // one reader, so all epilogue threads agree
      epi_bar();
      if (esh.flag) break;
      tc_fence_after();
      const uint32_t tb = trow + buf * BN;
      bool finish = whole;
      int first = g, last = g;
      if (!whole) {
        // park this segment's partial sum in the CTA's slot, then take a ticket
        const int side = (u == u0) ? 0 : 1;
        float* dst = a.partial + (static_cast<size_t>(g) * 2 + side) * slot_elems + r;
        for (int c0 = 0; c0 < BN; c0 += 16) {
          float v[16];
          tmem_ld16(tb + c0, v);
#pragma unroll
          for (int c = 0; c < 16; ++c) dst[static_cast<size_t>(c0 + c) * kTileN] = v[c];
        }
        first = cta_of(static_cast<long long>(t) * kb, a);
        last = cta_of(static_cast<long long>(t + 1) * kb - 1, a);
        __threadfence();
        epi_bar();
        if (r == 0) {
          const int tk = atomicAdd(a.tickets + t, 1);
          esh.flag = (tk == last - first);
          if (tk == last - first) a.tickets[t] = 0;
        }
        epi_bar();
        finish = esh.flag != 0;
        if (finish) __threadfence();
      }
      if (finish) {
        tile_rows_prepare<BN>(a, e, m0, r, esh);
        for (int c0 = 0; c0 < BN; c0 += 16) {
          float v[16];
          tmem_ld16(tb + c0, v);
          for (int o = first; o <= last; ++o) {
            if (o == g) continue;
            const int side_o = (unit_begin(o, a) / kb == t) ? 0 : 1;
            const float* src = a.partial + (static_cast<size_t>(o) * 2 + side_o) * slot_elems + r;
#pragma unroll
            for (int c = 0; c < 16; ++c) v[c] += __ldcg(src + static_cast<size_t>(c0 + c) * kTileN);
          }
          epilogue_chunk<BN>(a, rg, e, tn, m0, c0, r, v, stg, esh);
        }
        if (e.kind == EPI_ARGMAX) {
          // the CTA that finishes the last tile decodes the winning keys and resets them
          __threadfence();
          epi_bar();
          if (r == 0) {
            const int dn = atomicAdd(e.done, 1);
            esh.flag = (dn == a.n_tiles * a.m_tiles - 1);
          }
          epi_bar();
          if (esh.flag) {
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
          epi_bar();
        }
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
}

template <int BN>
cudaError_t launch_bn(const AMaps& amaps, const ARegions& rg, const CUtensorMap& xmap, const GemmArgs& a,
                      const GemmEpi& e, cudaStream_t stream) {
  using C = Cfg<BN>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t err = cudaFuncSetAttribute(gemm_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (err != cudaSuccess) return err;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemm_kernel<BN>, amaps, xmap, a, rg, e);
}

}  // namespace

int gemm_token_tile(int M) {
  if (M <= 16) return 16;
  if (M <= 32) return 32;
  if (M <= 64) return 64;
  if (M <= 128) return 128;
  return 256;
}

int gemm_grid(int M, int N, int K, int splits, size_t partial_elems, int num_sms) {
  const int BN = gemm_token_tile(M);
  const long long tiles = static_cast<long long>((N + kTileN - 1) / kTileN) * ((M + BN - 1) / BN);
  const int kb = (K + kTileK - 1) / kTileK;
  const long long units = tiles * kb;
  long long G = splits > 0 ? tiles * std::min(splits, kb) : num_sms;
  if (G > units) G = units;
  // 2 partial slots of 128 x BN floats per CTA, unless every CTA owns whole tiles
  const long long cap = static_cast<long long>(partial_elems / (2ull * kTileN * BN));
  if (G > cap && tiles % G != 0) {
    long long d = std::min<long long>(G, tiles);
    while (d > 1 && (tiles % d != 0) && d > cap) --d;
    while (d > 1 && tiles % d != 0) --d;
    G = d;
  }
  return static_cast<int>(std::max<long long>(G, 1));
}

cudaError_t launch_gemm(const AMaps& amaps, const ARegions& regions, const CUtensorMap& xmap, int M, int N, int K,
                        int splits, const GemmEpi& epi, const GemmWork& work, int num_sms, cudaStream_t stream) {
  if (M <= 0) return cudaSuccess;
  const int BN = gemm_token_tile(M);
  GemmArgs a{};
  a.M = M;
  a.N = N;
  a.K = K;
  a.k_blocks = (K + kTileK - 1) / kTileK;
  a.n_tiles = (N + kTileN - 1) / kTileN;
  a.m_tiles = (M + BN - 1) / BN;
  a.units = static_cast<long long>(a.n_tiles) * a.m_tiles * a.k_blocks;
  a.grid = gemm_grid(M, N, K, splits, work.partial_elems, num_sms);
  a.status = epi.status;
  a.partial = work.partial;
  a.tickets = work.tickets;
  if (static_cast<long long>(a.n_tiles) * a.m_tiles > work.n_tickets && a.grid % (a.n_tiles * a.m_tiles) != 0)
    return cudaErrorInvalidValue;
  switch (BN) {
    case 16: return launch_bn<16>(amaps, regions, xmap, a, epi, stream);
    case 32: return launch_bn<32>(amaps, regions, xmap, a, epi, stream);
    case 64: return launch_bn<64>(amaps, regions, xmap, a, epi, stream);
    case 128: return launch_bn<128>(amaps, regions, xmap, a, epi, stream);
    default: return launch_bn<256>(amaps, regions, xmap, a, epi, stream);
  }
}

}  // namespace dfl
