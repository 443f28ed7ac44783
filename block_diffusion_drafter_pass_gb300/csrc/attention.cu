// attention.cu - non-causal block attention over the injected context.
//
// For each sequence and kv head, the G*B query rows of the block (G query
// heads per kv head, B block positions) attend to every committed context key
// of that layer (paged, 64 tokens per page) and to the block's own B keys,
// with no mask (the drafter's attention is non-causal).
//
// The keys are split into chunks of whole 64-key tiles (flash-decoding). A
// persistent grid, one CTA per SM, walks the (sequence, kv head, chunk) work
// items. Per CTA:
//   warp 0     TMA producer: the item's queries once (two buffers, so the
//              next item's copies start while this one finishes), then per tile the key
//              rows [64][d] and the transposed value rows [d][64] of one page
//              (values are stored transposed in the pool so that both
//              products read K-major, 128-byte-swizzled operands);
//   warp 1     allocates tensor memory and issues tcgen05.mma from one
//              thread: S = Q K^T (M = 128 query rows, N = 64 keys) into one of
//              two TMEM S buffers, then O += P V (N = d) into the item's TMEM
//              O buffer, with P read from shared memory;
//   warps 2-5  one query row per thread (the TMEM lane quarter of the warp):
//              online softmax in the log2 domain on S read from TMEM, P
//              written to shared memory as bf16, O rescaled in TMEM only when
//              the row maximum grows by more than 2^8 (the stale maximum is a
//              valid reference point: P and O stay bounded by 256x).
// S_{t+1} is issued before P_t is ready, so the softmax of one tile overlaps
// the products of the next. Each item leaves an unnormalised partial (O,
// running max, running sum); attn_combine_kernel merges the chunks of a row.
// Query row r of an item is (block position j, head g of the group) with
// r = j*G + g (the order the 3D query box lands in shared memory).
#include <cuda.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace dfl {
namespace {

constexpr int kKeyTile = 64;
constexpr float kRescaleLog2 = 8.f;   // rescale O when the row max grows by more than 2^8

// Rows of the block's own key box: B rounded up to 16 or 32.
__host__ __device__ __forceinline__ int block_rows(int B) { return B <= 16 ? 16 : 32; }

template <int D>
struct ACfg {
  static constexpr int kStages = D == 128 ? 4 : 6;
  static constexpr int kBox = 64 * 128;                   // 64 rows x 128 bytes
  static constexpr int kKBytes = (D / 64) * kBox;         // keys [64][D]
  static constexpr int kVBytes = (D / 64) * kBox;         // values transposed [D][64]
  static constexpr int kStageBytes = kKBytes + kVBytes;
  static constexpr int kQBox = 128 * 128;                 // 128 query rows x 64 dims
  static constexpr int kQBytes = (D / 64) * kQBox;
  static constexpr int kPBytes = 128 * 128;               // P [128 rows][64 keys] bf16
  static constexpr int kSmem = kStages * kStageBytes + 2 * kQBytes + 2 * kPBytes + 1024;
  static constexpr uint32_t kTmemCols = D == 128 ? 512 : 256;   // S 2x64 + O 2xD
  static constexpr uint32_t kIdescS = idesc_bf16_f32(128, kKeyTile);
  static constexpr uint32_t kIdescO = idesc_bf16_f32(128, D);
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// 64 consecutive TMEM columns of this thread's lane (32x32b shape, x64).
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
      "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
        "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
        "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

// Store 32 consecutive TMEM columns of this thread's lane; completes with the
// tcgen05.wait::st in tmem_wait_st.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]), "f"(v[8]),
      "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]), "f"(v[15]), "f"(v[16]),
      "f"(v[17]), "f"(v[18]), "f"(v[19]), "f"(v[20]), "f"(v[21]), "f"(v[22]), "f"(v[23]), "f"(v[24]),
      "f"(v[25]), "f"(v[26]), "f"(v[27]), "f"(v[28]), "f"(v[29]), "f"(v[30]), "f"(v[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 16 lanes x 32 bits, two column halves: threads 0-15 read lanes 0-15 of the
// warp's quarter at columns [c, c+32), threads 16-31 the same lanes at
// columns [c+SPLIT, c+SPLIT+32).
template <int SPLIT>
__device__ __forceinline__ void tmem_ld_half32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.16x32bx2.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32], %33;\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr), "n"(SPLIT)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

template <int SPLIT>
__device__ __forceinline__ void tmem_st_half32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x32bx2.x32.b32 [%0], %33, {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]), "f"(v[8]),
      "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]), "f"(v[15]), "f"(v[16]),
      "f"(v[17]), "f"(v[18]), "f"(v[19]), "f"(v[20]), "f"(v[21]), "f"(v[22]), "f"(v[23]), "f"(v[24]),
      "f"(v[25]), "f"(v[26]), "f"(v[27]), "f"(v[28]), "f"(v[29]), "f"(v[30]), "f"(v[31]), "n"(SPLIT)
      : "memory");
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float m;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(m) : "f"(a), "f"(b), "f"(c));
  return m;
}

// Max of n values (n = 32 or 64) as independent three-input chains.
template <int N>
__device__ __forceinline__ float row_max(const float (&v)[N]) {
  float m0 = v[0], m1 = v[1], m2 = v[2], m3 = v[3];
#pragma unroll
  for (int c = 4; c + 8 <= N; c += 8) {
    m0 = max3(m0, v[c], v[c + 4]);
    m1 = max3(m1, v[c + 1], v[c + 5]);
    m2 = max3(m2, v[c + 2], v[c + 6]);
    m3 = max3(m3, v[c + 3], v[c + 7]);
  }
  m0 = max3(m0, v[N - 4], m1);
  m2 = max3(m2, v[N - 3], m3);
  return max3(m0, m2, max3(v[N - 2], v[N - 1], -INFINITY));
}

// Work decomposition shared by the three roles and the combine kernel.
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

struct Item {
  int i, kvh, tb, te;   // sequence index, kv head, tiles [tb, te)
};

// SPREAD (G*B <= 64): query row r sits in TMEM lane 32*(r/16) + r%16, so all
// four lane quarters (and the four SM sub-partitions that own them) carry 16
// rows, and two threads share a row (32 keys each). Otherwise one thread per
// row, row r in lane r.
template <int D, bool SPREAD>
__global__ void __launch_bounds__(192, 1)
    attn_kernel(const __grid_constant__ AttnMaps maps, const __grid_constant__ AttnArgs a) {
  using C = ACfg<D>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + S * C::kStageBytes;
  uint8_t* sP = sQ + 2 * C::kQBytes;   // queries double-buffered by item
  __shared__ __align__(8) uint64_t kv_full[S], kv_empty[S];
  __shared__ __align__(8) uint64_t q_full[2], q_empty[2], mma_done;
  __shared__ __align__(8) uint64_t s_full[2], p_full[2], pv_done[2], o_full[2], o_free[2];
  __shared__ uint32_t tmem_slot;
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
    for (int s = 0; s < S; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    mbar_init(&q_full[0], 1);
    mbar_init(&q_full[1], 1);
    mbar_init(&q_empty[0], 1);
    mbar_init(&q_empty[1], 1);
    mbar_init(&mma_done, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&p_full[b], 4);
      mbar_init(&pv_done[b], 1);
      mbar_init(&o_full[b], 1);
      mbar_init(&o_free[b], 4);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&maps.pool_k);
    tma_prefetch_desc(&maps.pool_vt);
    tma_prefetch_desc(&maps.q);
    tma_prefetch_desc(&maps.kblk);
    tma_prefetch_desc(&maps.vblk);
  }
  if (warp == 1) tmem_alloc(&tmem_slot, C::kTmemCols);
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
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  grid_dep_launch();
  const uint32_t tmem = tmem_slot;
  const int total = s_prefix[n_seq];

  auto decode = [&](int item) {
    Item it;
    int i = 0;
    while (i + 1 < n_seq && item >= s_prefix[i + 1]) ++i;
    const int local = item - s_prefix[i];
    it.i = i;
    it.kvh = local / s_nch[i];
    const int chunk = local - it.kvh * s_nch[i];
    it.tb = chunk * a.chunk_tiles;
    it.te = min(s_nctx[i] + 1, it.tb + a.chunk_tiles);
    return it;
  };
  auto give_up = [&]() {
    abort_flag = 1;
    latch_status(a.status, kDevTimeout);
  };

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      const int Bb = block_rows(B);
      int n = 0, k = 0;
      bool dead = false;
      for (int item = blockIdx.x; item < total && !dead; item += gridDim.x, ++k) {
        const Item it = decode(item);
        const int qb = k & 1;
        if (!mbar_wait(&q_empty[qb], ((k >> 1) & 1) ^ 1, &abort_flag)) {
          give_up();
          break;
        }
        uint8_t* qdst = sQ + qb * C::kQBytes;
        if constexpr (SPREAD) {
          // groups of 16 rows (gB positions x gG heads) to smem rows 32k .. 32k+15
          const int gG = a.q_group_heads, gB = 16 / gG, ng = (R + 15) / 16;
          mbar_arrive_expect_tx(&q_full[qb], ng * (D / 64) * 16 * 128);
          for (int g = 0; g < ng; ++g) {
            const int hpg = G / gG;                        // groups per block position
            const int j = g / hpg * gB, h0 = (g % hpg) * gG;
#pragma unroll
            for (int bx = 0; bx < D / 64; ++bx)
              tma_load_3d(qdst + bx * C::kQBox + g * 32 * 128, &maps.q, &q_full[qb], bx * 64, it.kvh * G + h0,
                          it.i * B + j);
          }
        } else {
          mbar_arrive_expect_tx(&q_full[qb], (D / 64) * R * 128);
#pragma unroll
          for (int bx = 0; bx < D / 64; ++bx)
            tma_load_3d(qdst + bx * C::kQBox, &maps.q, &q_full[qb], bx * 64, it.kvh * G, it.i * B);
        }
        const int slot = a.meta.slot[it.i];
        for (int t = it.tb; t < it.te; ++t, ++n) {
          const int s = n % S;
          if (!mbar_wait(&kv_empty[s], ((n / S) & 1) ^ 1, &abort_flag)) {
            give_up();
            dead = true;
            break;
          }
          uint8_t* ks = smem + s * C::kStageBytes;
          uint8_t* vs = ks + C::kKBytes;
          if (t < s_nctx[it.i]) {
            int page = -1;
            if (t < a.seqs.pages_per_seq) page = a.seqs.page_table[static_cast<size_t>(slot) * a.seqs.pages_per_seq + t];
            if (page < 0 || page >= a.pool_pages) {
              latch_status(a.status, kDevBounds);
              page = 0;
            }
            const int lp = a.layer * a.pool_pages + page;
            const int rowk = (lp * 2 * nkv + it.kvh) * kKeyTile;        // rows of d elements
            const int rowv = ((lp * 2 + 1) * nkv + it.kvh) * D;         // rows of 64 elements
            mbar_arrive_expect_tx(&kv_full[s], C::kStageBytes);
#pragma unroll
            for (int bx = 0; bx < D / 64; ++bx) {
              tma_load_2d(ks + bx * C::kBox, &maps.pool_k, &kv_full[s], bx * 64, rowk);
              tma_load_2d(vs + bx * C::kBox, &maps.pool_vt, &kv_full[s], 0, rowv + bx * 64);
            }
          } else {
            mbar_arrive_expect_tx(&kv_full[s], (D / 64) * Bb * 128 + C::kVBytes);
#pragma unroll
            for (int bx = 0; bx < D / 64; ++bx) {
              tma_load_3d(ks + bx * C::kBox, &maps.kblk, &kv_full[s], bx * 64, it.kvh, it.i * B);
              tma_load_2d(vs + bx * C::kBox, &maps.vblk, &kv_full[s], 0, (it.i * nkv + it.kvh) * D + bx * 64);
            }
          }
        }
      }
      // copies still in flight complete before shared memory is released
      for (int j = max(0, n - S); j < n; ++j) mbar_wait(&kv_full[j % S], (j / S) & 1);
      for (int j = max(0, k - 2); j < k; ++j) mbar_wait(&q_full[j & 1], (j >> 1) & 1);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t q_base = smem_u32(sQ), p_base = smem_u32(sP), kv_base = smem_u32(smem);
      auto issue_s = [&](int m, int qb) {   // S[m & 1] = Q K_m^T
        const uint32_t kb = kv_base + (m % S) * C::kStageBytes;
        const uint32_t qs = q_base + qb * C::kQBytes;
        const uint32_t d_tmem = tmem + (m & 1) * kKeyTile;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk & 3) * 32;   // 16 elements along K inside the 128-byte row
          tc_mma_bf16(d_tmem, sdesc_kmajor_sw128(qs + (kk >> 2) * C::kQBox + off),
                      sdesc_kmajor_sw128(kb + (kk >> 2) * C::kBox + off), C::kIdescS, kk > 0);
        }
        tc_commit(&s_full[m & 1]);
      };
      int n = 0, k = 0;
      bool dead = false;
      for (int item = blockIdx.x; item < total && !dead; item += gridDim.x, ++k) {
        const Item it = decode(item);
        const int nt = it.te - it.tb;
        const int ob = k & 1;
        const uint32_t o_tmem = tmem + 2 * kKeyTile + ob * D;
        const int qb = k & 1;
        if (!mbar_wait(&q_full[qb], (k >> 1) & 1, &abort_flag) ||
            !mbar_wait(&kv_full[n % S], (n / S) & 1, &abort_flag)) {
          give_up();
          break;
        }
        tc_fence_after();
        issue_s(n, qb);
        if (nt == 1) tc_commit(&q_empty[qb]);
        for (int lt = 0; lt < nt; ++lt) {
          const int m = n + lt;
          if (lt + 1 < nt) {
            if (!mbar_wait(&kv_full[(m + 1) % S], ((m + 1) / S) & 1, &abort_flag)) {
              give_up();
              dead = true;
              break;
            }
            tc_fence_after();
            issue_s(m + 1, qb);
            if (lt + 2 == nt) tc_commit(&q_empty[qb]);
          }
          if (!mbar_wait(&p_full[m & 1], (m >> 1) & 1, &abort_flag) ||
              (lt == 0 && !mbar_wait(&o_free[ob], ((k >> 1) & 1) ^ 1, &abort_flag))) {
            give_up();
            dead = true;
            break;
          }
          tc_fence_after();
          const uint32_t vb = kv_base + (m % S) * C::kStageBytes + C::kKBytes;
          const uint32_t pb = p_base + (m & 1) * C::kPBytes;
#pragma unroll
          for (int kk = 0; kk < kKeyTile / 16; ++kk)
            tc_mma_bf16(o_tmem, sdesc_kmajor_sw128(pb + kk * 32), sdesc_kmajor_sw128(vb + kk * 32), C::kIdescO,
                        (lt > 0 || kk > 0) ? 1u : 0u);
          tc_commit(&kv_empty[m % S]);
          tc_commit(&pv_done[m & 1]);
        }
        if (dead) break;
        tc_commit(&o_full[ob]);
        n += nt;
      }
      // every issued MMA completes before TMEM and shared memory are released
      tc_commit(&mma_done);
      mbar_wait(&mma_done, 0);
    }
  } else {
    // ---------------- softmax / output warps ----------------
    constexpr int kCols = SPREAD ? 32 : 64;                // S columns per thread
    const int quarter = warp & 3;                          // TMEM lanes 32*quarter .. +31
    const int half = SPREAD ? (lane >> 4) : 0;             // which 32 keys of the row (SPREAD)
    const int tlane = quarter * 32 + (SPREAD ? (lane & 15) : lane);   // TMEM lane = Q/P smem row
    const int row = SPREAD ? quarter * 16 + (lane & 15) : tlane;      // query row r
    const bool active = (SPREAD ? quarter * 16 : quarter * 32) < R;   // warp-uniform
    const uint32_t lane_tmem = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float sl2 = 1.4426950408889634f / sqrtf(static_cast<float>(D));   // log2(e)/sqrt(d)
    uint8_t* p_row = sP + tlane * 128;
    // waits taken by all 32 lanes together, so the warp-collective TMEM
    // accesses after them never diverge (also when a wait runs out)
    auto warp_wait = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, &abort_flag));
    };
    // O row of this thread: D columns (one thread per row) or D/2 (SPREAD)
    auto o_scale = [&](uint32_t o_tmem, float alpha) {
#pragma unroll
      for (int c0 = 0; c0 < (SPREAD ? D / 2 : D); c0 += 32) {
        float ov[32];
        if constexpr (SPREAD) tmem_ld_half32<D / 2>(o_tmem + c0, ov);
        else tmem_ld32(o_tmem + c0, ov);
#pragma unroll
        for (int c = 0; c < 32; ++c) ov[c] *= alpha;
        if constexpr (SPREAD) tmem_st_half32<D / 2>(o_tmem + c0, ov);
        else tmem_st32(o_tmem + c0, ov);
      }
      tmem_wait_st();
    };
    int n = 0, k = 0;
    bool dead = false;
    for (int item = blockIdx.x; item < total && !dead; item += gridDim.x, ++k) {
      const Item it = decode(item);
      const int nt = it.te - it.tb;
      const int ob = k & 1;
      const uint32_t o_tmem = lane_tmem + 2 * kKeyTile + ob * D;
      const int len = s_len[it.i];
      float m_run = -INFINITY, l_run = 0.f;   // l_run: this thread's share of the row sum
      for (int lt = 0; lt < nt; ++lt) {
        const int m = n + lt, b = m & 1;
        const int t = it.tb + lt;
        if (!warp_wait(&s_full[b], (m >> 1) & 1)) {
          give_up();
          dead = true;
          break;
        }
        tc_fence_after();
        if (active) {
          float sv[kCols];
          if constexpr (SPREAD) tmem_ld_half32<32>(lane_tmem + b * kKeyTile, sv);
          else tmem_ld64(lane_tmem + b * kKeyTile, sv);
          const int nvalid = t < s_nctx[it.i] ? min(kKeyTile, len - t * kKeyTile) : B;
          if (nvalid < kKeyTile) {   // warp-uniform: only a ragged last page or the block tile
            const int col0 = half * 32;
#pragma unroll
            for (int c = 0; c < kCols; ++c) sv[c] = col0 + c < nvalid ? sv[c] : -INFINITY;
          }
          float mx = row_max(sv);
          if constexpr (SPREAD) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          mx *= sl2;   // log2 units
          if (lt == 0) {
            m_run = mx;
          } else if (__any_sync(0xffffffffu, row < R && mx > m_run + kRescaleLog2)) {
            // O holds the products up to tile m-1: wait for them, then rescale
            if (!warp_wait(&pv_done[(m - 1) & 1], ((m - 1) >> 1) & 1)) {
              give_up();
              dead = true;
            }
            tc_fence_after();
            const float nm = fmaxf(m_run, mx);
            const float alpha = ex2(m_run - nm);
            l_run *= alpha;
            m_run = nm;
            if (!dead) o_scale(o_tmem, alpha);
          }
          float s4[4] = {0.f, 0.f, 0.f, 0.f};
          uint32_t pk[kCols / 2];
#pragma unroll
          for (int c = 0; c < kCols / 2; ++c) {
            const float p0 = ex2(fmaf(sv[2 * c], sl2, -m_run));
            const float p1 = ex2(fmaf(sv[2 * c + 1], sl2, -m_run));
            s4[c & 3] += p0 + p1;
            pk[c] = pack_bf16(p0, p1);
          }
          l_run += (s4[0] + s4[1]) + (s4[2] + s4[3]);
          // P buffer b was last read by the products of tile m-2
          if (!dead && !warp_wait(&pv_done[b], ((m >> 1) & 1) ^ 1)) {
            give_up();
            dead = true;
          }
          uint8_t* pr = p_row + b * C::kPBytes;
#pragma unroll
          for (int cc = 0; cc < kCols / 8; ++cc) {
            const int ch = half * 4 + cc;   // 16-byte chunk (8 keys) of the 128-byte P row
            *reinterpret_cast<uint4*>(pr + ((ch ^ (tlane & 7)) << 4)) =
                make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
          }
          fence_proxy_async_smem();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[b]);
        if (dead) break;
      }
      if (dead) break;
      if (!warp_wait(&o_full[ob], (k >> 1) & 1)) {
        give_up();
        break;
      }
      tc_fence_after();
      if (active) {
        if constexpr (SPREAD) l_run += __shfl_xor_sync(0xffffffffu, l_run, 16);
        const bool keep = row < R && item < a.items_cap;
        float* po = a.part_o + (static_cast<size_t>(item) * a.rows_pad + row) * D + half * (D / 2);
#pragma unroll
        for (int c0 = 0; c0 < (SPREAD ? D / 2 : D); c0 += 32) {
          float ov[32];
          if constexpr (SPREAD) tmem_ld_half32<D / 2>(o_tmem + c0, ov);
          else tmem_ld32(o_tmem + c0, ov);
          if (keep) {
#pragma unroll
            for (int c = 0; c < 32; c += 4)
              *reinterpret_cast<float4*>(po + c0 + c) = make_float4(ov[c], ov[c + 1], ov[c + 2], ov[c + 3]);
          }
        }
        if (keep && half == 0) a.part_ml[static_cast<size_t>(item) * a.rows_pad + row] = make_float2(m_run, l_run);
        if (row == 0 && half == 0 && item >= a.items_cap) latch_status(a.status, kDevBounds);   // host sizing prevents this
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&o_free[ob]);
      n += nt;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// Merge the chunks of each row: grid (n_q heads, n_seq, ceil(B/4)), one warp
// per (head, block position). Lanes split the chunks for the running max and
// sum, then read each chunk's partial row as one coalesced 16-byte-per-lane
// load (D = 128) and accumulate it with its weight exp2(m_c - M).
constexpr int kCombineWarps = 4;
constexpr int kCombineMaxChunks = 2048;

template <int D>
__global__ void __launch_bounds__(32 * kCombineWarps) attn_combine_kernel(const __grid_constant__ AttnArgs a) {
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
  const int r = j * G + gh;
  const size_t rp = static_cast<size_t>(a.rows_pad);
  float M = -INFINITY;
  for (int c = lane; c < nch; c += 32) M = fmaxf(M, a.part_ml[(base + c) * rp + r].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float L = 0.f;
  for (int c = lane; c < nch; c += 32) {
    const float2 ml = a.part_ml[(base + c) * rp + r];
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
  const float* po = a.part_o + (static_cast<size_t>(base) * rp + r) * D + lane * kPer;
  const size_t stride = rp * D;
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

template <int D, bool SPREAD>
cudaError_t launch_main(const AttnMaps& maps, const AttnArgs& a, int grid, cudaStream_t stream) {
  using C = ACfg<D>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e =
        cudaFuncSetAttribute(attn_kernel<D, SPREAD>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_pdl(attn_kernel<D, SPREAD>, dim3(grid), dim3(192), C::kSmem, stream, maps, a);
}

template <int D>
cudaError_t launch_d(const AttnMaps& maps, const AttnArgs& a, int grid, int part, cudaStream_t stream) {
  if (part == 0)
    return a.q_group_heads > 0 ? launch_main<D, true>(maps, a, grid, stream) : launch_main<D, false>(maps, a, grid, stream);
  return launch_pdl(attn_combine_kernel<D>,
                    dim3(a.n_q_heads, a.meta.n_seq, (a.meta.B + kCombineWarps - 1) / kCombineWarps),
                    dim3(32 * kCombineWarps), 0, stream, a);
}

}  // namespace

int attention_block_rows(int B) { return block_rows(B); }

int attention_spread_group(int G, int B) {
  if (G * B > 64) return 0;
  if (16 % G == 0) return G;
  if (G % 16 == 0) return 16;
  return 0;
}

int attention_ctas_per_sm(int head_dim) {
  int n = 0;
  auto q = [&](auto kern, int smem) {
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, 192, smem) != cudaSuccess) n = 1;
  };
  if (head_dim == 128) q(attn_kernel<128, true>, ACfg<128>::kSmem);
  else q(attn_kernel<64, true>, ACfg<64>::kSmem);
  return n < 1 ? 1 : n;
}

cudaError_t launch_attention(const AttnMaps& maps, const AttnArgs& a, int grid, int part, cudaStream_t stream) {
  const int G = a.n_q_heads / a.n_kv_heads, R = G * a.meta.B;
  if (R > 128 || a.rows_pad < R) return cudaErrorInvalidValue;
  if (a.q_group_heads > 0 && (R > 64 || attention_spread_group(G, a.meta.B) != a.q_group_heads))
    return cudaErrorInvalidValue;
  if (a.head_dim == 128) return launch_d<128>(maps, a, grid, part, stream);
  if (a.head_dim == 64) return launch_d<64>(maps, a, grid, part, stream);
  return cudaErrorInvalidValue;
}

}  // namespace dfl
