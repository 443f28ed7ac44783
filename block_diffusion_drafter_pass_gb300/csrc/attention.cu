// attention.cu - non-causal block attention over the injected context.
//
// For each sequence and kv head, the G*B query rows of the block (G query
// heads per kv head, B block positions) attend to every committed context key
// of that layer (paged, 64 tokens per page) and to the block's own B keys,
// with no mask (the drafter's attention is non-causal).
//
// The keys are split into chunks of whole 64-key tiles (flash-decoding). A
// persistent grid walks the (sequence, kv head, chunk) work items; per CTA
// one producer warp streams K/V tiles page by page with TMA (128-byte
// swizzle, STAGES-deep mbarrier ring) and the compute warps run
// QK^T and PV on tensor cores (mma.sync m16n8k16, bf16 in / fp32 accumulate)
// with an online softmax held in registers (warp-shuffle row max / sum).
// Each item leaves an unnormalised partial (O, running max, running sum);
// attn_combine_kernel merges the chunks of each row.
#include <cuda.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace dfl {
namespace {

constexpr int kStages = 3;
constexpr int kKeyTile = 64;

// Rows of the block's own K/V box: B rounded up to whole 16-key MMA steps.
__host__ __device__ __forceinline__ int block_rows(int B) { return B <= 16 ? 16 : 32; }

template <int D>
struct ACfg {
  static constexpr int kBox = kKeyTile * 64 * 2;          // one 64-key x 64-dim box, 8 KB
  static constexpr int kTileBytes = (D / 64) * kBox;      // K (or V) tile
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kSmem = kStages * kStageBytes + 1024;
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const uint32_t l = f32_to_bf16(lo), h = f32_to_bf16(hi);
  return l | (h << 16);
}

// Address of the 16-byte chunk `ch` (dims 8*ch..8*ch+7) of key row `key`
// inside a TMA-written tile of D/64 swizzled 64x64 boxes.
__device__ __forceinline__ uint32_t tile_addr(uint32_t base, int key, int ch) {
  return base + (ch >> 3) * (kKeyTile * 128) + key * 128 + (((ch & 7) ^ (key & 7)) << 4);
}

// Work decomposition shared by the producer, the compute warps and combine.
struct SeqSplit {
  int len;        // committed context tokens
  int n_ctx;      // context tiles
  int n_chunks;   // chunks (context tiles + the block tile)
};

__device__ __forceinline__ SeqSplit seq_split(const AttnArgs& a, int i) {
  SeqSplit s;
  s.len = a.seqs.len[a.meta.slot[i]];
  s.n_ctx = (s.len + kKeyTile - 1) / kKeyTile;
  s.n_chunks = (s.n_ctx + 1 + a.chunk_tiles - 1) / a.chunk_tiles;
  return s;
}

template <int D, int NCW>
__global__ void __launch_bounds__((NCW + 1) * 32, NCW <= 4 ? 2 : 1)
    attn_kernel(const __grid_constant__ CUtensorMap pool_map, const __grid_constant__ CUtensorMap kblk_map,
                const __grid_constant__ CUtensorMap vblk_map, const __grid_constant__ AttnArgs a) {
  using C = ACfg<D>;
  constexpr int kRowsPad = 16 * NCW;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full[kStages];
  __shared__ __align__(8) uint64_t empty[kStages];
  __shared__ int s_prefix[kMaxBatch + 1];
  __shared__ int s_len[kMaxBatch];
  __shared__ int s_nctx[kMaxBatch];
  __shared__ int s_nch[kMaxBatch];
  __shared__ volatile int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_seq = a.meta.n_seq, B = a.meta.B;
  const int nkv = a.n_kv_heads, G = a.n_q_heads / a.n_kv_heads;
  const int R = G * B;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NCW);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  grid_dep_wait();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int i = 0; i < n_seq; ++i) {
      const SeqSplit sp = seq_split(a, i);
      s_len[i] = sp.len;
      s_nctx[i] = sp.n_ctx;
      s_nch[i] = sp.n_chunks;
      s_prefix[i] = acc;
      acc += nkv * sp.n_chunks;
    }
    s_prefix[n_seq] = acc;
  }
  __syncthreads();
  grid_dep_launch();
  const int total = s_prefix[n_seq];

  if (warp == NCW) {
    // ---------------- producer ----------------
    if (lane == 0) {
      tma_prefetch_desc(&pool_map);
      const int Bb = block_rows(B);
      int it = 0;
      for (int item = blockIdx.x; item < total && !abort_flag; item += gridDim.x) {
        int i = 0;
        while (i + 1 < n_seq && item >= s_prefix[i + 1]) ++i;
        const int local = item - s_prefix[i];
        const int kvh = local / s_nch[i], chunk = local - kvh * s_nch[i];
        const int tb = chunk * a.chunk_tiles;
        const int te = min(s_nctx[i] + 1, tb + a.chunk_tiles);
        const int slot = a.meta.slot[i];
        for (int t = tb; t < te; ++t, ++it) {
          const int s = it % kStages;
          if (!mbar_wait(&empty[s], ((it / kStages) & 1) ^ 1, &abort_flag)) {
            abort_flag = 1;
            latch_status(a.status, kDevTimeout);
            break;
          }
          uint8_t* ks = smem + s * C::kStageBytes;
          uint8_t* vs = ks + C::kTileBytes;
          if (t < s_nctx[i]) {
            int page = -1;
            if (t < a.seqs.pages_per_seq) page = a.seqs.page_table[static_cast<size_t>(slot) * a.seqs.pages_per_seq + t];
            if (page < 0 || page >= a.pool_pages) {
              latch_status(a.status, kDevBounds);
              page = 0;
            }
            const int rowk = ((a.layer * a.pool_pages + page) * 2 * nkv + kvh) * kKeyTile;
            const int rowv = rowk + nkv * kKeyTile;
            mbar_arrive_expect_tx(&full[s], C::kStageBytes);
#pragma unroll
            for (int bx = 0; bx < D / 64; ++bx) {
              tma_load_2d(ks + bx * C::kBox, &pool_map, &full[s], bx * 64, rowk);
              tma_load_2d(vs + bx * C::kBox, &pool_map, &full[s], bx * 64, rowv);
            }
          } else {
            mbar_arrive_expect_tx(&full[s], 2 * (D / 64) * Bb * 128);
#pragma unroll
            for (int bx = 0; bx < D / 64; ++bx) {
              tma_load_3d(ks + bx * C::kBox, &kblk_map, &full[s], bx * 64, kvh, i * B);
              tma_load_3d(vs + bx * C::kBox, &vblk_map, &full[s], bx * 64, kvh, i * B);
            }
          }
        }
      }
      // drain copies still in flight (only matters after an abort)
      for (int j = max(0, it - kStages); j < it; ++j) mbar_wait(&full[j % kStages], (j / kStages) & 1);
    }
  } else {
    // ---------------- compute warps ----------------
    const int g = lane >> 2, tig = lane & 3;
    const float sl2 = 1.4426950408889634f / sqrtf(static_cast<float>(D));   // log2(e)/sqrt(d)
    const int rA = warp * 16 + g, rB = rA + 8;                               // this thread's two rows
    int it = 0;
    for (int item = blockIdx.x; item < total; item += gridDim.x) {
      if (abort_flag) break;
      int i = 0;
      while (i + 1 < n_seq && item >= s_prefix[i + 1]) ++i;
      const int local = item - s_prefix[i];
      const int kvh = local / s_nch[i], chunk = local - kvh * s_nch[i];
      const int tb = chunk * a.chunk_tiles;
      const int te = min(s_nctx[i] + 1, tb + a.chunk_tiles);
      const int len = s_len[i];

      // Q fragments for rows rA, rB (row r = g_head*B + j; zero beyond R)
      uint32_t qf[D / 16][4];
      {
        const uint16_t* qa = nullptr;
        const uint16_t* qb = nullptr;
        if (rA < R) qa = a.q + static_cast<size_t>(i * B + rA % B) * a.n_q_heads * D + static_cast<size_t>(kvh * G + rA / B) * D;
        if (rB < R) qb = a.q + static_cast<size_t>(i * B + rB % B) * a.n_q_heads * D + static_cast<size_t>(kvh * G + rB / B) * D;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const int c = kk * 16 + 2 * tig;
          qf[kk][0] = qa ? *reinterpret_cast<const uint32_t*>(qa + c) : 0u;
          qf[kk][1] = qb ? *reinterpret_cast<const uint32_t*>(qb + c) : 0u;
          qf[kk][2] = qa ? *reinterpret_cast<const uint32_t*>(qa + c + 8) : 0u;
          qf[kk][3] = qb ? *reinterpret_cast<const uint32_t*>(qb + c + 8) : 0u;
        }
      }
      float o[D / 8][4];
#pragma unroll
      for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
      float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;

      bool dead = false;
      for (int t = tb; t < te; ++t, ++it) {
        const int s = it % kStages;
        if (!mbar_wait(&full[s], (it / kStages) & 1, &abort_flag)) {
          abort_flag = 1;
          latch_status(a.status, kDevTimeout);
          dead = true;
          break;
        }
        const int nvalid = t < s_nctx[i] ? min(kKeyTile, len - t * kKeyTile) : B;
        const uint32_t kbase = smem_u32(smem + s * C::kStageBytes);
        const uint32_t vbase = kbase + C::kTileBytes;

        // S = Q K^T over 64 keys (8 n-tiles of 8 keys)
        float sc[8][4];
#pragma unroll
        for (int n = 0; n < 8; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
        const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
          for (int np = 0; np < 4; ++np) {
            const int key = np * 16 + ((mi >> 1) << 3) + rr;
            const int ch = kk * 2 + (mi & 1);
            uint32_t b0, b1, b2, b3;
            ldsm_x4(tile_addr(kbase, key, ch), b0, b1, b2, b3);
            mma_bf16(sc[2 * np], qf[kk], b0, b1);
            mma_bf16(sc[2 * np + 1], qf[kk], b2, b3);
          }
        }
        // online softmax (log2 domain)
        float mxA = -INFINITY, mxB = -INFINITY;
#pragma unroll
        for (int n = 0; n < 8; ++n) {
          const int k0 = n * 8 + 2 * tig;
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const bool ok = (k0 + e) < nvalid;
            sc[n][e] = ok ? sc[n][e] * sl2 : -INFINITY;
            sc[n][2 + e] = ok ? sc[n][2 + e] * sl2 : -INFINITY;
            mxA = fmaxf(mxA, sc[n][e]);
            mxB = fmaxf(mxB, sc[n][2 + e]);
          }
        }
        mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 1));
        mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 2));
        mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 1));
        mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 2));
        const float nmA = fmaxf(mA, mxA), nmB = fmaxf(mB, mxB);
        const float alA = exp2f(mA - nmA), alB = exp2f(mB - nmB);   // exp2(-inf) = 0 on the first tile
        float sumA = 0.f, sumB = 0.f;
#pragma unroll
        for (int n = 0; n < 8; ++n) {
          sc[n][0] = exp2f(sc[n][0] - nmA);
          sc[n][1] = exp2f(sc[n][1] - nmA);
          sc[n][2] = exp2f(sc[n][2] - nmB);
          sc[n][3] = exp2f(sc[n][3] - nmB);
          sumA += sc[n][0] + sc[n][1];
          sumB += sc[n][2] + sc[n][3];
        }
        sumA += __shfl_xor_sync(0xffffffffu, sumA, 1);
        sumA += __shfl_xor_sync(0xffffffffu, sumA, 2);
        sumB += __shfl_xor_sync(0xffffffffu, sumB, 1);
        sumB += __shfl_xor_sync(0xffffffffu, sumB, 2);
        lA = lA * alA + sumA;
        lB = lB * alB + sumB;
        mA = nmA;
        mB = nmB;
#pragma unroll
        for (int n = 0; n < D / 8; ++n) {
          o[n][0] *= alA;
          o[n][1] *= alA;
          o[n][2] *= alB;
          o[n][3] *= alB;
        }
        // O += P V over the valid 16-key steps
        const int ksteps = (nvalid + 15) >> 4;
#pragma unroll
        for (int k2 = 0; k2 < 4; ++k2) {
          if (k2 < ksteps) {
            uint32_t pa[4];
            pa[0] = pack_bf16(sc[2 * k2][0], sc[2 * k2][1]);
            pa[1] = pack_bf16(sc[2 * k2][2], sc[2 * k2][3]);
            pa[2] = pack_bf16(sc[2 * k2 + 1][0], sc[2 * k2 + 1][1]);
            pa[3] = pack_bf16(sc[2 * k2 + 1][2], sc[2 * k2 + 1][3]);
#pragma unroll
            for (int dp = 0; dp < D / 16; ++dp) {
              const int key = k2 * 16 + ((mi & 1) << 3) + rr;
              const int ch = dp * 2 + (mi >> 1);
              uint32_t b0, b1, b2, b3;
              ldsm_x4_t(tile_addr(vbase, key, ch), b0, b1, b2, b3);
              mma_bf16(o[2 * dp], pa, b0, b1);
              mma_bf16(o[2 * dp + 1], pa, b2, b3);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
      }
      if (dead) break;
      if (item >= a.items_cap) {   // the host sizes the split so this cannot happen
        if (lane == 0) latch_status(a.status, kDevBounds);
        continue;
      }
      // unnormalised partial of this item
      float* po = a.part_o + static_cast<size_t>(item) * kRowsPad * D;
#pragma unroll
      for (int n = 0; n < D / 8; ++n) {
        const int c = n * 8 + 2 * tig;
        *reinterpret_cast<float2*>(po + static_cast<size_t>(rA) * D + c) = make_float2(o[n][0], o[n][1]);
        *reinterpret_cast<float2*>(po + static_cast<size_t>(rB) * D + c) = make_float2(o[n][2], o[n][3]);
      }
      if (tig == 0) {
        a.part_ml[static_cast<size_t>(item) * kRowsPad + rA] = make_float2(mA, lA);
        a.part_ml[static_cast<size_t>(item) * kRowsPad + rB] = make_float2(mB, lB);
      }
    }
  }
  __syncthreads();
}

// Merge the chunks of each row: grid (n_q heads, n_seq, ceil(B/4)), one warp
// per (head, block row). Lanes split the chunks for the running max and sum,
// then read each chunk's partial row as one coalesced 16-byte-per-lane load
// (D = 128) and accumulate it with its weight exp2(m_c - M).
constexpr int kCombineWarps = 4;
constexpr int kCombineMaxChunks = 2048;

template <int D, int NCW>
__global__ void __launch_bounds__(32 * kCombineWarps) attn_combine_kernel(const __grid_constant__ AttnArgs a) {
  constexpr int kRowsPad = 16 * NCW;
  constexpr int kPer = D / 32;                 // dims per lane: 4 (D = 128) or 2 (D = 64)
  __shared__ float wsm[kCombineWarps][kCombineMaxChunks];
  grid_dep_wait();
  grid_dep_launch();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hq = blockIdx.x, i = blockIdx.y;
  const int j = blockIdx.z * kCombineWarps + warp;
  const int B = a.meta.B;
  const int nkv = a.n_kv_heads, G = a.n_q_heads / nkv;
  const int kvh = hq / G, gh = hq - kvh * G;
  int base = 0;
  for (int s = 0; s < i; ++s) base += nkv * seq_split(a, s).n_chunks;
  const int nch = seq_split(a, i).n_chunks;
  base += kvh * nch;
  if (j >= B || base + nch > a.items_cap || nch > kCombineMaxChunks) {
    if (j < B && lane == 0) latch_status(a.status, kDevBounds);
    return;
  }
  const int r = gh * B + j;
  float M = -INFINITY;
  for (int c = lane; c < nch; c += 32) M = fmaxf(M, a.part_ml[static_cast<size_t>(base + c) * kRowsPad + r].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float L = 0.f;
  for (int c = lane; c < nch; c += 32) {
    const float2 ml = a.part_ml[static_cast<size_t>(base + c) * kRowsPad + r];
    const float w = exp2f(ml.x - M);
    wsm[warp][c] = w;
    L += w * ml.y;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  __syncwarp();
  float acc[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
  const float* po = a.part_o + (static_cast<size_t>(base) * kRowsPad + r) * D + lane * kPer;
  const size_t stride = static_cast<size_t>(kRowsPad) * D;
  int c = 0;
  for (; c + 4 <= nch; c += 4) {
    float v[4][kPer];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if constexpr (kPer == 4) {
        const float4 t = __ldcg(reinterpret_cast<const float4*>(po + (c + u) * stride));
        v[u][0] = t.x; v[u][1] = t.y; v[u][2] = t.z; v[u][3] = t.w;
      } else {
        const float2 t = __ldcg(reinterpret_cast<const float2*>(po + (c + u) * stride));
        v[u][0] = t.x; v[u][1] = t.y;
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int e = 0; e < kPer; ++e) acc[e] += wsm[warp][c + u] * v[u][e];
  }
  for (; c < nch; ++c)
#pragma unroll
    for (int e = 0; e < kPer; ++e) acc[e] += wsm[warp][c] * __ldcg(po + c * stride + e);
  const float inv = 1.f / L;
  uint16_t* out = a.out + static_cast<size_t>(i * B + j) * a.n_q_heads * D + static_cast<size_t>(hq) * D + lane * kPer;
#pragma unroll
  for (int e = 0; e < kPer; ++e) out[e] = f32_to_bf16(acc[e] * inv);
}

template <int D, int NCW>
cudaError_t launch_dn(const CUtensorMap& pm, const CUtensorMap& km, const CUtensorMap& vm, const AttnArgs& a,
                      int grid, int part, cudaStream_t stream) {
  using C = ACfg<D>;
  if (part == 0) {
    static bool attr_set = false;
    if (!attr_set) {
      cudaError_t e =
          cudaFuncSetAttribute(attn_kernel<D, NCW>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
      if (e != cudaSuccess) return e;
      attr_set = true;
    }
    return launch_pdl(attn_kernel<D, NCW>, dim3(grid), dim3((NCW + 1) * 32), C::kSmem, stream, pm, km, vm, a);
  }
  return launch_pdl(attn_combine_kernel<D, NCW>,
                    dim3(a.n_q_heads, a.meta.n_seq, (a.meta.B + kCombineWarps - 1) / kCombineWarps),
                    dim3(32 * kCombineWarps), 0, stream, a);
}

}  // namespace

int attention_block_rows(int B) { return block_rows(B); }

int attention_ctas_per_sm(int head_dim, int ncw) {
  int n = 0;
  auto q = [&](auto kern, int threads, int smem) {
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, threads, smem) != cudaSuccess) n = 1;
  };
  if (head_dim == 128) {
    if (ncw <= 1) q(attn_kernel<128, 1>, 64, ACfg<128>::kSmem);
    else if (ncw <= 2) q(attn_kernel<128, 2>, 96, ACfg<128>::kSmem);
    else if (ncw <= 4) q(attn_kernel<128, 4>, 160, ACfg<128>::kSmem);
    else q(attn_kernel<128, 8>, 288, ACfg<128>::kSmem);
  } else {
    if (ncw <= 1) q(attn_kernel<64, 1>, 64, ACfg<64>::kSmem);
    else if (ncw <= 2) q(attn_kernel<64, 2>, 96, ACfg<64>::kSmem);
    else if (ncw <= 4) q(attn_kernel<64, 4>, 160, ACfg<64>::kSmem);
    else q(attn_kernel<64, 8>, 288, ACfg<64>::kSmem);
  }
  return n < 1 ? 1 : n;
}

cudaError_t launch_attention(const CUtensorMap& pool_map, const CUtensorMap& kblk_map, const CUtensorMap& vblk_map,
                             const AttnArgs& a, int grid, int part, cudaStream_t stream) {
  const int R = (a.n_q_heads / a.n_kv_heads) * a.meta.B;
  const int ncw = (R + 15) / 16;
  if (a.head_dim == 128) {
    if (ncw <= 1) return launch_dn<128, 1>(pool_map, kblk_map, vblk_map, a, grid, part, stream);
    if (ncw <= 2) return launch_dn<128, 2>(pool_map, kblk_map, vblk_map, a, grid, part, stream);
    if (ncw <= 4) return launch_dn<128, 4>(pool_map, kblk_map, vblk_map, a, grid, part, stream);
    if (ncw <= 8) return launch_dn<128, 8>(pool_map, kblk_map, vblk_map, a, grid, part, stream);
  } else if (a.head_dim == 64) {
    if (ncw <= 1) return launch_dn<64, 1>(pool_map, kblk_map, vblk_map, a, grid, part, stream);
    if (ncw <= 2) return launch_dn<64, 2>(pool_map, kblk_map, vblk_map, a, grid, part, stream);
    if (ncw <= 4) return launch_dn<64, 4>(pool_map, kblk_map, vblk_map, a, grid, part, stream);
    if (ncw <= 8) return launch_dn<64, 8>(pool_map, kblk_map, vblk_map, a, grid, part, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace dfl
