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
  static constexpr int kTmemCols = BN < 32 ? 32 : BN;
  static constexpr int kSmem = kStages * kStageBytes + 1024;
};

struct GemmArgs {
  int M, N, K;
  int k_blocks, kb_per_split, splits;
  int n_tiles, m_tiles;
  int n_pad;           // row pitch of the split-K partial buffer
  float* partial;
  int* tickets;
  int* status;
};

struct EpiShared {
  unsigned long long cand[4][16];
  int col_pos[16];
  int col_dst[16];     // KV_APPEND: pool row index of (page, slot) without layer/kv/head
  int flag;
};

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

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
      const bool ok = (n < a.N) && (m0 + c0 + c < a.M);
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
  if (r < 16) {
    const int m = m0 + c0 + r;
    int pos = -1, dst = -1;
    if (m < a.M) {
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
    sh.col_pos[r] = pos;
    sh.col_dst[r] = dst;
  }
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
      const int pos = sh.col_pos[c];
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
        const int dst = sh.col_dst[c];
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

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ AMaps amaps, const __grid_constant__ CUtensorMap xmap,
                const __grid_constant__ GemmArgs a, const __grid_constant__ ARegions rg,
                const __grid_constant__ GemmEpi e) {
  using C = Cfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full[C::kStages];
  __shared__ __align__(8) uint64_t empty[C::kStages];
  __shared__ __align__(8) uint64_t accum;
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;
  __shared__ EpiShared esh;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int split = blockIdx.x % a.splits;
  const int tile_n = blockIdx.x / a.splits;
  const int tile_m = blockIdx.y;
  const int kb0 = split * a.kb_per_split;
  const int nkb = min(a.kb_per_split, a.k_blocks - kb0);
  const int m0 = tile_m * BN;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&accum, 1);
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

  // Wait for the producer of our activations (programmatic dependent launch).
  grid_dep_wait();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      int map_lo, map_hi, row_lo, row_hi;
      if (rg.paired) {
        map_lo = 0; map_hi = 1;
        row_lo = row_hi = tile_n * 64;
      } else {
        const int reg = region_of(rg, tile_n);
        map_lo = map_hi = reg;
        row_lo = (tile_n - rg.tile_begin[reg]) * kTileN;
        row_hi = row_lo + 64;
      }
      const uint64_t wpol = policy_evict_first();
      int issued = 0;
      for (int i = 0; i < nkb; ++i) {
        const int s = i % C::kStages;
        const uint32_t ph = (i / C::kStages) & 1;
        if (!mbar_wait(&empty[s], ph ^ 1, &abort_flag)) {
          abort_flag = 1;
          latch_status(a.status, kDevTimeout);
          break;
        }
        uint8_t* sa = smem + s * C::kStageBytes;
        uint8_t* sb = sa + kABytes;
        const int kx = (kb0 + i) * kTileK;
        mbar_arrive_expect_tx(&full[s], C::kStageBytes);
        tma_load_2d_hint(sa, &amaps.m[map_lo], &full[s], kx, row_lo, wpol);
        tma_load_2d_hint(sa + kABytes / 2, &amaps.m[map_hi], &full[s], kx, row_hi, wpol);
        tma_load_2d(sb, &xmap, &full[s], kx, m0);
        ++issued;
      }
      // On abort, drain copies still in flight before shared memory is released.
      if (abort_flag) {
        for (int i = max(0, issued - C::kStages); i < issued; ++i)
          mbar_wait(&full[i % C::kStages], (i / C::kStages) & 1);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      constexpr uint32_t idesc = idesc_bf16_f32(kTileN, BN);
      for (int i = 0; i < nkb; ++i) {
        const int s = i % C::kStages;
        const uint32_t ph = (i / C::kStages) & 1;
        if (!mbar_wait(&full[s], ph, &abort_flag)) {
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
          tc_mma_bf16(tmem, ad + 2 * k, bd + 2 * k, idesc, (i | k) != 0 ? 1u : 0u);
        tc_commit(&empty[s]);
      }
      tc_commit(&accum);
    }
  } else {
    // ---------------- epilogue warps ----------------
    const int q = warp & 3;                 // TMEM lane quarter of this warp
    const int r = q * 32 + lane;            // tile row = output feature
    float* stg = reinterpret_cast<float*>(smem);
    const uint32_t trow = tmem + (static_cast<uint32_t>(q * 32) << 16);
    bool ok = mbar_wait(&accum, 0, &abort_flag);
    if (!ok) {
      abort_flag = 1;
      latch_status(a.status, kDevTimeout);
    }
    epi_bar();
    ok = ok && !abort_flag && nkb > 0;
    tc_fence_after();
    bool last = true;
    const int tile_id = tile_m * a.n_tiles + tile_n;
    if (ok && a.splits > 1) {
      // write this split's partial tile, then take a ticket
      const int n = tile_n * kTileN + r;
      float* dst = a.partial + (static_cast<size_t>(split) * a.m_tiles * BN + m0) * a.n_pad + n;
      for (int c0 = 0; c0 < BN; c0 += 16) {
        float v[16];
        tmem_ld16(trow + c0, v);
#pragma unroll
        for (int c = 0; c < 16; ++c) dst[static_cast<size_t>(c0 + c) * a.n_pad] = v[c];
      }
      __threadfence();
      epi_bar();
      if (r == 0) {
        const int t = atomicAdd(a.tickets + tile_id, 1);
        esh.flag = (t == a.splits - 1);
        if (t == a.splits - 1) a.tickets[tile_id] = 0;
      }
      epi_bar();
      last = esh.flag != 0;
      if (last) __threadfence();
    }
    if (ok && last) {
      for (int c0 = 0; c0 < BN; c0 += 16) {
        float v[16];
        tmem_ld16(trow + c0, v);
        if (a.splits > 1) {
          const int n = tile_n * kTileN + r;
          for (int s = 0; s < a.splits; ++s) {
            if (s == split) continue;
            const float* src = a.partial + (static_cast<size_t>(s) * a.m_tiles * BN + m0 + c0) * a.n_pad + n;
#pragma unroll
            for (int c = 0; c < 16; ++c) v[c] += __ldcg(src + static_cast<size_t>(c) * a.n_pad);
          }
        }
        epilogue_chunk<BN>(a, rg, e, tile_n, m0, c0, r, v, stg, esh);
      }
      if (e.kind == EPI_ARGMAX) {
        // the last tile to finish decodes the winning keys and resets them
        __threadfence();
        epi_bar();
        if (r == 0) {
          const int t = atomicAdd(e.done, 1);
          esh.flag = (t == a.n_tiles * a.m_tiles - 1);
        }
        epi_bar();
        if (esh.flag) {
          __threadfence();
          for (int m = r; m < a.M; m += 128) {
            const unsigned long long k = atomicExch(e.keys + m, 0ull);
            e.out_ids[m] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(k & 0xFFFFFFFFull));
            if (e.out_logit) e.out_logit[m] = ordered_key_inv(static_cast<uint32_t>(k >> 32));
          }
          if (r == 0) *e.done = 0;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  grid_dep_launch();
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
  dim3 grid(a.n_tiles * a.splits, a.m_tiles);
  gemm_kernel<BN><<<grid, kThreads, C::kSmem, stream>>>(amaps, xmap, a, rg, e);
  return cudaGetLastError();
}

}  // namespace

int gemm_token_tile(int M) {
  if (M <= 16) return 16;
  if (M <= 32) return 32;
  if (M <= 64) return 64;
  if (M <= 128) return 128;
  return 256;
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
  a.n_pad = a.n_tiles * kTileN;
  a.status = epi.status;
  const int tiles = a.n_tiles * a.m_tiles;
  if (splits <= 0) {
    splits = 1;
    if (tiles < num_sms) splits = num_sms / tiles;
    if (splits > a.k_blocks) splits = a.k_blocks;
    if (splits > 16) splits = 16;
  }
  if (splits > a.k_blocks) splits = a.k_blocks;
  if (splits < 1) splits = 1;
  while (splits > 1 && (static_cast<size_t>(splits) * a.m_tiles * BN * a.n_pad > work.partial_elems ||
                        tiles > work.n_tickets))
    --splits;
  a.kb_per_split = (a.k_blocks + splits - 1) / splits;
  a.splits = (a.k_blocks + a.kb_per_split - 1) / a.kb_per_split;
  a.partial = work.partial;
  a.tickets = work.tickets;
  switch (BN) {
    case 16: return launch_bn<16>(amaps, regions, xmap, a, epi, stream);
    case 32: return launch_bn<32>(amaps, regions, xmap, a, epi, stream);
    case 64: return launch_bn<64>(amaps, regions, xmap, a, epi, stream);
    case 128: return launch_bn<128>(amaps, regions, xmap, a, epi, stream);
    default: return launch_bn<256>(amaps, regions, xmap, a, epi, stream);
  }
}

}  // namespace dfl
