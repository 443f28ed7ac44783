// path_selector.cu - the DFlash 2 path selector after the drafter pass
// ("DFlash 2" notes, "Solution - Lightweight Path Selector").
//
// The drafter keeps the 16 largest logits U_t of every masked position t as
// its candidates C_t; every adjacent pair (a in C_{t-1}, b in C_t) is scored
//
//     S_t(a, b) = U_t(b) + < A(a) * H(h_t), B(b) >
//
// and a greedy walk from the anchor picks one candidate per position. A and
// B are linear maps of the token embedding (A = W_A E, B = W_B E), so both are
// token-indexed tables computed once when the selector is installed: one fp32
// row of 512 values per token, A in [0, 256) and B in [256, 512). H(h_t) =
// W_H h~_t comes out of the LM-head GEMM as 256 extra output features of the
// final-normalised row.
//
// Per draft pass (after the LM-head GEMM stored logits and H as fp32):
//   sel_topk_kernel   CTA (slice, row): the 16 largest (logit, column) keys
//                     of one column slice of one draft row;
//   sel_pairs_kernel  CTA (position t, sequence): merges the slice lists of
//                     rows t and t-1 into C_t and C_{t-1}, stages A of the
//                     predecessors and B of the candidates in shared memory
//                     and scores all 16 x 16 pairs; the last CTA of a
//                     sequence to finish (atomic ticket, nothing spins) walks
//                     the score matrices and writes the draft ids.
// Keys order logits as floats (-0 folded onto +0) and put the lower column
// first among equal logits; the walk takes the first maximum, i.e. the
// higher-ranked candidate among equal scores.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace dfl {
namespace {

constexpr int kTopThreads = 256;
constexpr int kTopQ = 8;                                  // float4 per thread
constexpr int kSliceCols = kTopThreads * 4 * kTopQ;       // 8192 columns per CTA
constexpr int kTopCandCap = 8 * 16 * 4 * kTopQ;           // 8 warps x 16 lanes x 32 keys
constexpr int kPairThreads = 512;
constexpr int kPadRow = kSelDim + 1;   // shared-memory row pitch (bank spread)
static_assert(kSliceCols == kSelSliceCols, "slice width");
static_assert(kSelDim == 256, "H(h_t) is loaded by one thread per dimension of the first 256");
static_assert(2 * 2 * kSelMaxSlices * kSelK * 8 <= 2 * kSelK * kPadRow * 4, "merge lists fit the staging buffer");
static_assert(kMaxBlock * kSelK * kSelK <= 2 * kSelK * kPadRow, "the walk's scores fit the staging buffer");

// Order-preserving 64-bit key of (logit, column): larger logit first, lower
// column first among equal logits. 0 never arises from a number and marks an
// empty entry.
__device__ __forceinline__ unsigned long long logit_key(float v, int col) {
  uint32_t b = __float_as_uint(v == 0.f ? 0.f : v);
  b = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return (static_cast<unsigned long long>(b) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(col));
}

__device__ __forceinline__ float key_value(unsigned long long k) {
  uint32_t b = static_cast<uint32_t>(k >> 32);
  b = (b & 0x80000000u) ? (b & 0x7FFFFFFFu) : ~b;
  return __uint_as_float(b);
}

__device__ __forceinline__ int key_col(unsigned long long k) {
  return static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(k));
}

// Logits row of draft row r (block row j = 1 + r % T of sequence r / T).
__device__ __forceinline__ size_t draft_logit_row(int r, int B) {
  const int T = B - 1;
  return static_cast<size_t>(r / T) * B + 1 + r % T;
}

// Exact top-16 of m distinct nonzero keys in shared memory by counting: a
// key's rank is the number of larger keys. Threads tid, tid + nthr, ... take
// one key each; out[rank] for ranks below 16, zeros past m.
__device__ __forceinline__ void top_by_rank(const unsigned long long* keys, int m, int tid, int nthr,
                                            unsigned long long* out) {
  for (int j = tid; j < m; j += nthr) {
    const unsigned long long k = keys[j];
    int rank = 0;
    for (int q = 0; q < m; ++q) rank += keys[q] > k;
    if (rank < kSelK) out[rank] = k;
  }
  if (tid >= m && tid < kSelK) out[tid] = 0;
}

// Order-preserving unsigned image of a float (for integer max on floats).
__device__ __forceinline__ uint32_t ordered_bits(float v) {
  const uint32_t b = __float_as_uint(v);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// CTA (slice, row): the 16 largest keys of columns [s * kSliceCols, +kSliceCols)
// of draft row r. Every thread holds kTopQ float4 of the slice.
// Threshold: in every warp two lanes reach the warp's second largest lane
// maximum, so 16 values of the CTA reach the smallest of the 8 warps' second
// largest lane maxima and every value below it is out. Values at or above it
// (about 30 per CTA for unordered data; ties can add more) are appended as
// keys and ranked exactly. If ties overflow the buffer, the slice is redone
// with exact keys: the warp's 16th largest lane-maximum key bounds it, and at
// most 16 lanes x 32 keys per warp reach that.
__global__ void __launch_bounds__(kTopThreads, 4) sel_topk_kernel(const float* __restrict__ logits, int ld, int V,
                                                                  int B, unsigned long long* __restrict__ part) {
  __shared__ unsigned long long s_cand[kTopCandCap];
  __shared__ unsigned long long s_tau_key;
  __shared__ uint32_t s_r2[kTopThreads / 32];
  __shared__ int s_m;
  grid_dep_wait();
  grid_dep_launch();
  const int s = blockIdx.x, r = blockIdx.y, slices = gridDim.x;
  const int tid = threadIdx.x, lane = tid & 31;
  if (tid == 0) {
    s_tau_key = 0;
    s_m = 0;
  }
  const float* row = logits + draft_logit_row(r, B) * ld;
  const int c0 = s * kSliceCols, c1 = min(V, c0 + kSliceCols);
  // columns c0 + 4 (tid + 256 u) + e; whole float4 below c1 lie below the
  // row's padded width (a multiple of 128); columns past c1 read as -inf and
  // are masked where keys are formed
  float4 v[kTopQ];
#pragma unroll
  for (int u = 0; u < kTopQ; ++u) {
    const int c = c0 + 4 * (tid + kTopThreads * u);
    v[u] = c < c1 ? __ldcs(reinterpret_cast<const float4*>(row + c)) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
  }
  // lane maximum (fmaxf skips NaN; an all-NaN lane counts as -inf, which
  // only loosens the bound)
  float bv = -INFINITY;
#pragma unroll
  for (int u = 0; u < kTopQ; ++u) bv = fmaxf(bv, fmaxf(fmaxf(v[u].x, v[u].y), fmaxf(v[u].z, v[u].w)));
  if (bv != bv) bv = -INFINITY;
  const uint32_t ob = ordered_bits(bv == 0.f ? 0.f : bv);
  const uint32_t m1 = __reduce_max_sync(0xffffffffu, ob);
  const int l1 = __ffs(__ballot_sync(0xffffffffu, ob == m1)) - 1;
  const uint32_t m2 = __reduce_max_sync(0xffffffffu, lane == l1 ? 0u : ob);
  if (lane == 0) s_r2[tid >> 5] = m2;
  __syncthreads();   // s_r2, s_tau_key, s_m
  uint32_t tb = s_r2[0];
#pragma unroll
  for (int w = 1; w < kTopThreads / 32; ++w) tb = min(tb, s_r2[w]);
  const float tau = __uint_as_float((tb & 0x80000000u) ? (tb & 0x7FFFFFFFu) : ~tb);
  auto key_at = [&](float x, int c) -> unsigned long long {
    return (c < c1 && x == x) ? logit_key(x, c) : 0ull;
  };
#pragma unroll
  for (int u = 0; u < kTopQ; ++u) {
    const int c = c0 + 4 * (tid + kTopThreads * u);
    const float x4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (x4[e] >= tau) {   // -0 and +0 compare equal; NaN never passes
        const unsigned long long k = key_at(x4[e], c + e);
        if (k != 0) {
          const int at = atomicAdd(&s_m, 1);
          if (at < kTopCandCap) s_cand[at] = k;
        }
      }
    }
  }
  __syncthreads();
  if (s_m > kTopCandCap) {   // ties at the threshold: exact keys (the slice is read again)
    const int n_local = kTopQ * 4;
    unsigned long long best = 0;
    for (int q = 0; q < n_local; ++q) {
      const int c = c0 + 4 * (tid + kTopThreads * (q >> 2)) + (q & 3);
      if (c < c1) best = max(best, key_at(row[c], c));
    }
    int kr = 0;
    for (int o = 1; o < 32; ++o) kr += __shfl_sync(0xffffffffu, best, (lane + o) & 31) > best;
    __syncthreads();   // every thread has read s_m
    if (tid == 0) s_m = 0;
    if (kr == kSelK - 1) atomicMax(&s_tau_key, best);
    __syncthreads();
    const unsigned long long tk = s_tau_key;   // 0 when no warp has 16 lanes with keys: all keys kept
    for (int q = 0; q < n_local; ++q) {
      const int c = c0 + 4 * (tid + kTopThreads * (q >> 2)) + (q & 3);
      const unsigned long long k = c < c1 ? key_at(row[c], c) : 0ull;
      if (k != 0 && k >= tk) s_cand[atomicAdd(&s_m, 1)] = k;
    }
    __syncthreads();
  }
  top_by_rank(s_cand, s_m, tid, kTopThreads, part + (static_cast<size_t>(r) * slices + s) * kSelK);
}

struct PairsArgs {
  const unsigned long long* part;   // [rows][slices][kSelK] slice lists
  int slices;
  const float* logits;              // [n_seq*B][ld]: logits, then H(h_t) at column h_col
  int ld, h_col, V, B;
  const float* table;               // [V][2 * kSelDim]: A | B rows per token
  const int32_t* anchors;           // [n_seq]
  float* scores;                    // [n_seq][T][kSelK][kSelK]
  int32_t* cand;                    // [n_seq][T][kSelK]
  float* cand_u;                    // [n_seq][T][kSelK]
  int32_t* next;                    // [n_seq][T][kSelK] pick at t after predecessor rank a
  float* top_logit;                 // [n_seq][T] the largest logit of each row
  int* tickets;                     // [n_seq], zero between launches
  int32_t* draft_ids;               // [n_seq][T]
  int* status;
};

__global__ void __launch_bounds__(kPairThreads) sel_pairs_kernel(const __grid_constant__ PairsArgs a) {
  // [0]: A(a) * H(h_t) of the predecessors, [1]: B(b) of the candidates;
  // before that the merge's key lists, after it the walk's score matrices
  __shared__ __align__(16) float s_buf[2][kSelK][kPadRow];
  __shared__ int s_cd[kMaxBlock * kSelK];
  __shared__ float s_h[kSelDim];
  __shared__ int s_pred[kSelK], s_cand[kSelK];
  __shared__ float s_u[kSelK];
  __shared__ unsigned long long s_top[2][kSelK];
  __shared__ unsigned long long s_tau[2];
  __shared__ int s_m[2];
  __shared__ int s_last;
  float(&s_ah)[kSelK][kPadRow] = s_buf[0];
  float(&s_b)[kSelK][kPadRow] = s_buf[1];
  grid_dep_wait();
  grid_dep_launch();
  const int t = blockIdx.x, i = blockIdx.y, T = a.B - 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_pred = t == 0 ? 1 : kSelK;
  const size_t row = static_cast<size_t>(i) * a.B + 1 + t;
  // Merge the slice lists: threads [0, 256) take draft row t, [256, 512) row
  // t-1. A slice list's 16th key bounds the row's 16th largest from below, so
  // only keys at or above the largest such bound are ranked.
  const int half = threadIdx.x >> 8, ht = threadIdx.x & 255;
  const int n_keys = a.slices * kSelK;   // <= kSelMaxSlices * 16 = 1024
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(&s_buf[0][0][0]) + half * 2 * kSelMaxSlices * kSelK;
  unsigned long long* kept = keys + kSelMaxSlices * kSelK;
  const bool merging = half == 0 || t > 0;
  if (threadIdx.x < 2) {
    s_tau[threadIdx.x] = 0;
    s_m[threadIdx.x] = 0;
  }
  if (merging) {   // all loads in flight before the stores
    const unsigned long long* src = a.part + static_cast<size_t>(i * T + t - half) * n_keys;
    unsigned long long kv[kSelMaxSlices * kSelK / 256];
#pragma unroll
    for (int u = 0; u < kSelMaxSlices * kSelK / 256; ++u) kv[u] = ht + 256 * u < n_keys ? __ldcg(src + ht + 256 * u) : 0ull;
#pragma unroll
    for (int u = 0; u < kSelMaxSlices * kSelK / 256; ++u)
      if (ht + 256 * u < n_keys) keys[ht + 256 * u] = kv[u];
  }
  if (half == 0) s_h[ht] = a.logits[row * a.ld + a.h_col + ht];
  __syncthreads();
  if (merging && ht < a.slices) atomicMax(&s_tau[half], keys[ht * kSelK + kSelK - 1]);
  __syncthreads();
  if (merging) {
    const unsigned long long tau = s_tau[half];
    for (int q = ht; q < n_keys; q += 256) {
      const unsigned long long k = keys[q];
      if (k != 0 && k >= tau) kept[atomicAdd(&s_m[half], 1)] = k;
    }
  }
  __syncthreads();
  if (merging) top_by_rank(kept, s_m[half], ht, 256, s_top[half]);
  __syncthreads();
  if (threadIdx.x < kSelK) {
    const unsigned long long k = s_top[0][threadIdx.x];
    int c = key_col(k);
    if (k == 0 || c < 0 || c >= a.V) {
      latch_status(a.status, kDevBounds);
      c = 0;
    }
    s_cand[threadIdx.x] = c;
    s_u[threadIdx.x] = k ? key_value(k) : -INFINITY;
  } else if (threadIdx.x < 2 * kSelK) {
    const int q = threadIdx.x - kSelK;
    if (t > 0) {
      const unsigned long long k = s_top[1][q];
      int c = key_col(k);
      if (k == 0 || c < 0 || c >= a.V) c = 0;   // reported by the CTA that owns row t-1
      s_pred[q] = c;
    } else if (q == 0) {
      int c = a.anchors[i];
      if (c < 0 || c >= a.V) {
        latch_status(a.status, kDevBounds);
        c = 0;
      }
      s_pred[0] = c;
    }
  }
  __syncthreads();
  // stage A(pred) * H and B(cand): 16 rows of 256 each, float4 loads, all
  // four of a thread in flight before the stores
  {
    constexpr int kQuads = kSelK * kSelDim / 4;   // 1024 float4 per matrix
    constexpr int kPer = 2 * kQuads / kPairThreads;
    float4 tv[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int q = threadIdx.x + kPairThreads * u;
      const int which = q / kQuads, rr = (q % kQuads) / (kSelDim / 4), d4 = (q % (kSelDim / 4)) * 4;
      const int tok = which == 0 ? (rr < n_pred ? s_pred[rr] : -1) : s_cand[rr];
      tv[u] = tok >= 0 ? __ldg(reinterpret_cast<const float4*>(a.table + static_cast<size_t>(tok) * (2 * kSelDim) +
                                                               which * kSelDim + d4))
                       : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int q = threadIdx.x + kPairThreads * u;
      const int which = q / kQuads, rr = (q % kQuads) / (kSelDim / 4), d4 = (q % (kSelDim / 4)) * 4;
      if (which == 0) {
        s_ah[rr][d4 + 0] = tv[u].x * s_h[d4 + 0];
        s_ah[rr][d4 + 1] = tv[u].y * s_h[d4 + 1];
        s_ah[rr][d4 + 2] = tv[u].z * s_h[d4 + 2];
        s_ah[rr][d4 + 3] = tv[u].w * s_h[d4 + 3];
      } else {
        s_b[rr][d4 + 0] = tv[u].x;
        s_b[rr][d4 + 1] = tv[u].y;
        s_b[rr][d4 + 2] = tv[u].z;
        s_b[rr][d4 + 3] = tv[u].w;
      }
    }
  }
  __syncthreads();
  // warp = predecessor a; lane = candidate b (lane & 15) and half (lane >> 4)
  // of the dimensions: half h takes d = 32j + 16h + q, so the two halves read
  // disjoint banks of the padded rows
  const size_t sbase = (static_cast<size_t>(i) * T + t) * kSelK;
  if (warp < n_pred) {
    const int b = lane & 15, h = lane >> 4;
    float acc = 0.f;
#pragma unroll 4
    for (int j = 0; j < kSelDim / 32; ++j) {
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const int d = 32 * j + 16 * h + q;
        acc = fmaf(s_ah[warp][d], s_b[b][d], acc);
      }
    }
    acc += __shfl_xor_sync(0xffffffffu, acc, 16);
    // lanes l and l ^ 16 hold the same score; the walk's step from
    // predecessor a is the first maximum over b
    float sv = s_u[b] + acc;
    if (sv != sv) sv = -INFINITY;
    const uint32_t ob = ordered_bits(sv == 0.f ? 0.f : sv);
    const uint32_t mx = __reduce_max_sync(0xffffffffu, ob);
    const int best = __ffs(__ballot_sync(0xffffffffu, ob == mx)) - 1;
    if (lane < kSelK) a.scores[(sbase + warp) * kSelK + lane] = sv;
    if (lane == 0) a.next[sbase + warp] = best;
  }
  if (threadIdx.x < kSelK) {
    a.cand[sbase + threadIdx.x] = s_cand[threadIdx.x];
    a.cand_u[sbase + threadIdx.x] = s_u[threadIdx.x];
  }
  if (threadIdx.x == 0 && a.top_logit) a.top_logit[static_cast<size_t>(i) * T + t] = s_u[0];
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(a.tickets + i, 1) == T - 1;
  }
  __syncthreads();
  if (!s_last) return;
  // The last CTA of sequence i: gather the T steps (the pick after each
  // predecessor) and candidate lists, then follow the picks from the anchor.
  __threadfence();
  const size_t c0 = static_cast<size_t>(i) * T * kSelK;
  {
    const int q = threadIdx.x;
    const int nx = q < T * kSelK ? __ldcg(a.next + c0 + q) : 0;
    const int id = q < T * kSelK ? __ldcg(a.cand + c0 + q) : 0;
    if (q < T * kSelK) {
      s_cd[q] = id;
      reinterpret_cast<int*>(&s_buf[0][0][0])[q] = nx;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const int* nx = reinterpret_cast<const int*>(&s_buf[0][0][0]);
    int p = 0;   // rank of the predecessor (the anchor at t = 0)
    for (int tt = 0; tt < T; ++tt) {
      p = nx[tt * kSelK + p] & (kSelK - 1);
      a.draft_ids[static_cast<size_t>(i) * T + tt] = s_cd[tt * kSelK + p];
    }
    a.tickets[i] = 0;
  }
}

}  // namespace

cudaError_t launch_path_select(const SelectArgs& s, cudaStream_t stream) {
  if (s.n_seq <= 0 || s.B < 2) return cudaSuccess;
  const int T = s.B - 1, rows = s.n_seq * T;
  cudaError_t e = launch_pdl(sel_topk_kernel, dim3(s.slices, rows), dim3(kTopThreads), 0, stream, s.logits, s.ld,
                             s.V, s.B, s.part);
  if (e != cudaSuccess) return e;
  PairsArgs a;
  a.part = s.part;
  a.slices = s.slices;
  a.logits = s.logits;
  a.ld = s.ld;
  a.h_col = s.h_col;
  a.V = s.V;
  a.B = s.B;
  a.table = s.table;
  a.anchors = s.anchors;
  a.scores = s.scores;
  a.cand = s.cand;
  a.cand_u = s.cand_u;
  a.next = s.next;
  a.top_logit = s.top_logit;
  a.tickets = s.tickets;
  a.draft_ids = s.draft_ids;
  a.status = s.status;
  return launch_pdl(sel_pairs_kernel, dim3(T, s.n_seq), dim3(kPairThreads), 0, stream, a);
}

}  // namespace dfl
