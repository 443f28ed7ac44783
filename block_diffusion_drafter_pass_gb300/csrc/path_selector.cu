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
//   topk_slices_kernel (topk.cuh) CTA (slice, row): the 16 largest (logit,
//                     column) keys of one 8192-column slice of one draft row;
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
#include "topk.cuh"

namespace dfl {
namespace {

constexpr int kPairThreads = 512;
constexpr int kPadRow = kSelDim + 1;   // shared-memory row pitch (bank spread)
using topk::key_col;
using topk::key_value;
using topk::ordered_bits;
static_assert(topk::In<float>::kSliceCols == kSelSliceCols, "slice width");
static_assert(kSelDim == 256, "H(h_t) is loaded by one thread per dimension of the first 256");
static_assert(2 * 2 * kSelMaxSlices * kSelK * 8 <= 2 * kSelK * kPadRow * 4, "merge lists fit the staging buffer");
static_assert(kMaxBlock * kSelK * kSelK <= 2 * kSelK * kPadRow, "the walk's scores fit the staging buffer");

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
  __shared__ unsigned long long s_tau[2], s_lo[2];
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
  // t-1 (nothing at t = 0, though they join the barriers).
  const int half = threadIdx.x >> 8, ht = threadIdx.x & 255;
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(&s_buf[0][0][0]) + half * 2 * kSelMaxSlices * kSelK;
  unsigned long long* kept = keys + kSelMaxSlices * kSelK;
  const bool merging = half == 0 || t > 0;
  if (half == 0) s_h[ht] = a.logits[row * a.ld + a.h_col + ht];
  topk::merge_lists<kSelK>(a.part + static_cast<size_t>(i * T + t - (merging ? half : 0)) * a.slices * kSelK,
                           merging ? a.slices : 0, ht, 256, keys, kept, &s_tau[half], &s_lo[half], &s_m[half],
                           s_top[half],
                           [] { __syncthreads(); });
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
  cudaError_t e = launch_pdl(topk::topk_slices_kernel<float, kSelK, true>, dim3(s.slices, rows), dim3(topk::kThreads), 0,
                             stream, s.logits, s.ld,
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
