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
constexpr int kPairThreads = 512;
constexpr int kPadRow = kSelDim + 1;   // shared-memory row pitch (bank spread)

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

// t[] sorted in decreasing order; keeps the kSelK largest of t and k.
__device__ __forceinline__ void top_insert(unsigned long long (&t)[kSelK], unsigned long long k) {
  if (k <= t[kSelK - 1]) return;
  t[kSelK - 1] = k;
#pragma unroll
  for (int i = kSelK - 1; i > 0; --i) {
    const unsigned long long hi = t[i] > t[i - 1] ? t[i] : t[i - 1];
    const unsigned long long lo = t[i] > t[i - 1] ? t[i - 1] : t[i];
    t[i - 1] = hi;
    t[i] = lo;
  }
}

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w > v ? w : v;
  }
  return v;
}

// Every lane holds a decreasing list t[]; returns, in lane k < kSelK, the
// k-th largest key of the warp's union (0 where fewer exist). Keys are
// distinct, so each round's maximum leaves exactly one lane's list.
__device__ __forceinline__ unsigned long long warp_top(unsigned long long (&t)[kSelK]) {
  const int lane = threadIdx.x & 31;
  unsigned long long mine = 0;
  for (int k = 0; k < kSelK; ++k) {
    const unsigned long long m = warp_max_u64(t[0]);
    if (lane == k) mine = m;
    if (m != 0 && t[0] == m) {
#pragma unroll
      for (int i = 0; i + 1 < kSelK; ++i) t[i] = t[i + 1];
      t[kSelK - 1] = 0;
    }
  }
  return mine;
}

// Logits row of draft row r (block row j = 1 + r % T of sequence r / T).
__device__ __forceinline__ size_t draft_logit_row(int r, int B) {
  const int T = B - 1;
  return static_cast<size_t>(r / T) * B + 1 + r % T;
}

__global__ void __launch_bounds__(kTopThreads) sel_topk_kernel(const float* __restrict__ logits, int ld, int V,
                                                               int B, int slice_cols,
                                                               unsigned long long* __restrict__ part) {
  __shared__ unsigned long long wtop[kTopThreads / 32][kSelK];
  grid_dep_wait();
  grid_dep_launch();
  const int s = blockIdx.x, r = blockIdx.y, slices = gridDim.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* row = logits + draft_logit_row(r, B) * ld;
  const int c0 = s * slice_cols, c1 = min(V, c0 + slice_cols);
  unsigned long long t[kSelK];
#pragma unroll
  for (int i = 0; i < kSelK; ++i) t[i] = 0;
  // float4 body (c0 and the row pitch are multiples of 4 floats), four loads
  // in flight per thread, then the ragged tail
  const int n4 = c1 > c0 ? (c1 - c0) >> 2 : 0;
  const float4* p4 = reinterpret_cast<const float4*>(row + c0);
  int i = threadIdx.x;
  for (; i + 3 * kTopThreads < n4; i += 4 * kTopThreads) {
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = __ldcs(p4 + i + u * kTopThreads);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int c = c0 + 4 * (i + u * kTopThreads);
      top_insert(t, logit_key(v[u].x, c));
      top_insert(t, logit_key(v[u].y, c + 1));
      top_insert(t, logit_key(v[u].z, c + 2));
      top_insert(t, logit_key(v[u].w, c + 3));
    }
  }
  for (; i < n4; i += kTopThreads) {
    const float4 v = __ldcs(p4 + i);
    const int c = c0 + 4 * i;
    top_insert(t, logit_key(v.x, c));
    top_insert(t, logit_key(v.y, c + 1));
    top_insert(t, logit_key(v.z, c + 2));
    top_insert(t, logit_key(v.w, c + 3));
  }
  for (int c = c0 + 4 * n4 + threadIdx.x; c < c1; c += kTopThreads) top_insert(t, logit_key(row[c], c));
  const unsigned long long w = warp_top(t);
  if (lane < kSelK) wtop[warp][lane] = w;
  __syncthreads();
  if (warp == 0) {
    // lane l takes entries 4l .. 4l+3 of the warps' lists (consecutive
    // entries of one warp's decreasing list)
    const unsigned long long* flat = &wtop[0][0];
#pragma unroll
    for (int q = 0; q < kSelK; ++q) t[q] = q < 4 ? flat[4 * lane + q] : 0ull;
    const unsigned long long k = warp_top(t);
    if (lane < kSelK) part[(static_cast<size_t>(r) * slices + s) * kSelK + lane] = k;
  }
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
  float* top_logit;                 // [n_seq][T] the largest logit of each row
  int* tickets;                     // [n_seq], zero between launches
  int32_t* draft_ids;               // [n_seq][T]
  int* status;
};

// Merge the slice lists of draft row r into its kSelK candidates (one warp).
__device__ __forceinline__ unsigned long long merge_row(const PairsArgs& a, int r) {
  const int lane = threadIdx.x & 31;
  unsigned long long t[kSelK];
  const unsigned long long* src = a.part + (static_cast<size_t>(r) * a.slices + lane) * kSelK;
  if (lane < a.slices) {
    const ulonglong2* s2 = reinterpret_cast<const ulonglong2*>(src);
#pragma unroll
    for (int q = 0; q < kSelK / 2; ++q) {
      const ulonglong2 v = __ldcg(s2 + q);
      t[2 * q] = v.x;
      t[2 * q + 1] = v.y;
    }
  } else {
#pragma unroll
    for (int q = 0; q < kSelK; ++q) t[q] = 0;
  }
  return warp_top(t);
}

__global__ void __launch_bounds__(kPairThreads) sel_pairs_kernel(const __grid_constant__ PairsArgs a) {
  // [0]: A(a) * H(h_t) of the predecessors, [1]: B(b) of the candidates;
  // the walk reuses the whole array for a sequence's T score matrices
  __shared__ float s_buf[2][kSelK][kPadRow];
  __shared__ int s_cd[kMaxBlock * kSelK];
  __shared__ float s_h[kSelDim];
  __shared__ int s_pred[kSelK], s_cand[kSelK];
  __shared__ float s_u[kSelK];
  __shared__ int s_last;
  float(&s_ah)[kSelK][kPadRow] = s_buf[0];
  float(&s_b)[kSelK][kPadRow] = s_buf[1];
  grid_dep_wait();
  grid_dep_launch();
  const int t = blockIdx.x, i = blockIdx.y, T = a.B - 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_pred = t == 0 ? 1 : kSelK;
  const size_t row = static_cast<size_t>(i) * a.B + 1 + t;
  if (warp == 0) {
    const unsigned long long k = merge_row(a, i * T + t);
    if (lane < kSelK) {
      int c = key_col(k);
      if (k == 0 || c < 0 || c >= a.V) {
        latch_status(a.status, kDevBounds);
        c = 0;
      }
      s_cand[lane] = c;
      s_u[lane] = k ? key_value(k) : -INFINITY;
    }
  } else if (warp == 1) {
    if (t > 0) {
      const unsigned long long k = merge_row(a, i * T + t - 1);
      if (lane < kSelK) {
        int c = key_col(k);
        if (k == 0 || c < 0 || c >= a.V) c = 0;   // reported by the CTA that owns row t-1
        s_pred[lane] = c;
      }
    } else if (lane == 0) {
      int c = a.anchors[i];
      if (c < 0 || c >= a.V) {
        latch_status(a.status, kDevBounds);
        c = 0;
      }
      s_pred[0] = c;
    }
  } else if (warp >= 8) {
    const int d = threadIdx.x - 256;
    s_h[d] = a.logits[row * a.ld + a.h_col + d];
  }
  __syncthreads();
  // stage A(pred) * H and B(cand): 16 rows of 256 each, float4 loads
  {
    constexpr int kQuads = kSelK * kSelDim / 4;   // 1024 float4 per matrix
#pragma unroll
    for (int q = threadIdx.x; q < 2 * kQuads; q += kPairThreads) {
      const int which = q / kQuads, rr = (q % kQuads) / (kSelDim / 4), d4 = (q % (kSelDim / 4)) * 4;
      if (which == 0 && rr >= n_pred) continue;
      const int tok = which == 0 ? s_pred[rr] : s_cand[rr];
      const float4 v = __ldg(reinterpret_cast<const float4*>(a.table + static_cast<size_t>(tok) * (2 * kSelDim) +
                                                            which * kSelDim + d4));
      if (which == 0) {
        s_ah[rr][d4 + 0] = v.x * s_h[d4 + 0];
        s_ah[rr][d4 + 1] = v.y * s_h[d4 + 1];
        s_ah[rr][d4 + 2] = v.z * s_h[d4 + 2];
        s_ah[rr][d4 + 3] = v.w * s_h[d4 + 3];
      } else {
        s_b[rr][d4 + 0] = v.x;
        s_b[rr][d4 + 1] = v.y;
        s_b[rr][d4 + 2] = v.z;
        s_b[rr][d4 + 3] = v.w;
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
    if (lane < kSelK) a.scores[(sbase + warp) * kSelK + lane] = s_u[lane] + acc;
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
  // The last CTA of sequence i: gather its T score matrices (T * 256 <=
  // 31 * 256 floats, within s_buf) and candidate lists, then walk.
  __threadfence();
  float* sc = &s_buf[0][0][0];
  int* cd = s_cd;
  const size_t s0 = static_cast<size_t>(i) * T * kSelK * kSelK;
  for (int q = threadIdx.x; q < T * kSelK * kSelK; q += kPairThreads) sc[q] = __ldcg(a.scores + s0 + q);
  for (int q = threadIdx.x; q < T * kSelK; q += kPairThreads)
    cd[q] = __ldcg(a.cand + static_cast<size_t>(i) * T * kSelK + q);
  __syncthreads();
  if (warp == 0) {
    int p = 0;   // rank of the predecessor (the anchor at t = 0)
    for (int tt = 0; tt < T; ++tt) {
      int b = lane & 15;
      float v = sc[(tt * kSelK + p) * kSelK + b];
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, v, o);
        const int ob = __shfl_xor_sync(0xffffffffu, b, o);
        if (ov > v || (ov == v && ob < b)) {
          v = ov;
          b = ob;
        }
      }
      p = b;
      if (lane == 0) a.draft_ids[static_cast<size_t>(i) * T + tt] = cd[tt * kSelK + p];
    }
    if (lane == 0) a.tickets[i] = 0;
  }
}

}  // namespace

cudaError_t launch_path_select(const SelectArgs& s, cudaStream_t stream) {
  if (s.n_seq <= 0 || s.B < 2) return cudaSuccess;
  const int T = s.B - 1, rows = s.n_seq * T;
  cudaError_t e = launch_pdl(sel_topk_kernel, dim3(s.slices, rows), dim3(kTopThreads), 0, stream, s.logits, s.ld,
                             s.V, s.B, s.slice_cols, s.part);
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
  a.top_logit = s.top_logit;
  a.tickets = s.tickets;
  a.draft_ids = s.draft_ids;
  a.status = s.status;
  return launch_pdl(sel_pairs_kernel, dim3(T, s.n_seq), dim3(kPairThreads), 0, stream, a);
}

}  // namespace dfl
