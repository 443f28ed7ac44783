// topk.cuh - the K largest logits of long rows (K = 16 or 32), shared by the
// path selector (top-16 candidates) and temperature sampling (top-k filter).
//
// Keys order (logit, column) pairs: a larger logit first, the lower column
// first among equal logits (-0 and +0 are one value). A key is 64 bits: the
// order-preserving image of the float above the complemented column; 0 never
// arises from a number and marks an empty entry. NaN is never a candidate.
//
// Pass 1, topk_slices_kernel: one CTA of 256 threads per 8192-column slice of
// a row, each thread holding 32 fp32 or bf16 values of the slice in registers.
// Threshold: in every warp, R = K / 8 lanes reach the warp's R-th largest lane
// maximum, so K values of the CTA reach the smallest of the 8 warps' R-th
// largest lane maxima and every value below it is out. The values at or above
// it (a few dozen per slice for unordered data) are appended as keys to a
// shared buffer and ranked exactly by counting. Ties can overflow the
// buffer (all-equal logits): then the buffer's K-th largest key, larger than
// the current bound since the buffer holds more than K distinct keys at or
// above it, becomes the bound and the slice is scanned again, until the keys
// at or above the bound fit.
// Pass 2 (merge_lists, called by the consuming kernel): the keys at or above
// a lower bound of the row's K-th largest key are ranked by counting; the
// bound is the larger of the slices' largest K-th key and the smallest c-th
// key, c = ceil(K / slices).
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace dfl {
namespace topk {

constexpr int kThreads = 256;
constexpr int kCandCap = 4096;                          // shared key buffer

template <typename InT>
struct In;
template <>
struct In<float> {
  static constexpr int kPerLoad = 4;
  static constexpr int kQuads = 8;                                 // 16-byte loads per thread: 32 values
  static constexpr int kMinBlocks = 4;                             // CTAs per SM (64 registers)
  static constexpr int kSliceCols = kThreads * kQuads * kPerLoad;   // 8192
};
template <>
struct In<uint16_t> {
  static constexpr int kPerLoad = 8;
  static constexpr int kQuads = 4;                                 // 32 values per thread
  static constexpr int kMinBlocks = 4;
  static constexpr int kSliceCols = kThreads * kQuads * kPerLoad;   // 8192
};

__device__ __forceinline__ uint32_t ordered_bits(float v) {
  const uint32_t b = __float_as_uint(v);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float from_ordered(uint32_t b) {
  return __uint_as_float((b & 0x80000000u) ? (b & 0x7FFFFFFFu) : ~b);
}

__device__ __forceinline__ unsigned long long logit_key(float v, int col) {
  return (static_cast<unsigned long long>(ordered_bits(v == 0.f ? 0.f : v)) << 32) |
         (0xFFFFFFFFu - static_cast<uint32_t>(col));
}

__device__ __forceinline__ float key_value(unsigned long long k) { return from_ordered(static_cast<uint32_t>(k >> 32)); }

__device__ __forceinline__ int key_col(unsigned long long k) {
  return static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(k));
}

// Exact top-K of m distinct nonzero keys in shared memory by counting: a
// key's rank is the number of larger keys. out[rank] for ranks below K,
// zeros past m. Threads tid, tid + nthr, ... take one key each.
template <int K>
__device__ __forceinline__ void top_by_rank(const unsigned long long* keys, int m, int tid, int nthr,
                                            unsigned long long* out) {
  for (int j = tid; j < m; j += nthr) {
    const unsigned long long k = keys[j];
    int rank = 0;
#pragma unroll 8
    for (int q = 0; q < m; ++q) rank += keys[q] > k;
    if (rank < K) out[rank] = k;
  }
  if (tid >= m && tid < K) out[tid] = 0;
}

// Logits row of list row r: draft rows skip each block's anchor row.
template <bool kDraftRows>
__device__ __forceinline__ size_t logit_row(int r, int B) {
  if constexpr (kDraftRows) {
    const int T = B - 1;
    return static_cast<size_t>(r / T) * B + 1 + r % T;
  } else {
    return static_cast<size_t>(r);
  }
}

template <typename InT>
__device__ __forceinline__ float elem(const uint4 (&v)[In<InT>::kQuads], int q) {
  if constexpr (In<InT>::kPerLoad == 4) {
    const uint32_t w = (&v[q >> 2].x)[q & 3];
    return __uint_as_float(w);
  } else {
    const uint32_t w = (&v[q >> 3].x)[(q & 7) >> 1];
    return __uint_as_float((q & 1) ? (w & 0xFFFF0000u) : (w << 16));
  }
}

// Largest value of one 16-byte load (NaN skipped): fp32 maxima, or packed
// bf16x2 maxima for bf16 (exact, -0 and +0 equal).
template <typename InT>
__device__ __forceinline__ float load_max(const uint4& w) {
  if constexpr (In<InT>::kPerLoad == 4) {
    return fmaxf(fmaxf(__uint_as_float(w.x), __uint_as_float(w.y)), fmaxf(__uint_as_float(w.z), __uint_as_float(w.w)));
  } else {
    const __nv_bfloat162 m = __hmax2(__hmax2(*reinterpret_cast<const __nv_bfloat162*>(&w.x),
                                             *reinterpret_cast<const __nv_bfloat162*>(&w.y)),
                                     __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&w.z),
                                             *reinterpret_cast<const __nv_bfloat162*>(&w.w)));
    return fmaxf(__bfloat162float(m.x), __bfloat162float(m.y));
  }
}

// CTA (slice, row) -> part[(row * slices + slice) * K + i], the slice's K
// largest keys in decreasing order (zeros when it holds fewer).
// Rows have pitch ld elements; whole 16-byte loads below the row's last valid
// column stay within the row (ld and V multiples of the load width).
template <typename InT, int K, bool kDraftRows>
__global__ void __launch_bounds__(kThreads, In<InT>::kMinBlocks) topk_slices_kernel(const InT* __restrict__ logits, int ld, int V,
                                                                  int B, unsigned long long* __restrict__ part) {
  constexpr int kQuads = In<InT>::kQuads, kPer = In<InT>::kPerLoad, kSlice = In<InT>::kSliceCols;
  constexpr int kVals = kQuads * kPer;
  constexpr int R = K / 8;
  static_assert(K % 8 == 0 && R >= 1 && R <= 4, "K of 8, 16, 24 or 32");
  __shared__ unsigned long long s_cand[kCandCap];
  __shared__ uint32_t s_rw[kThreads / 32];
  __shared__ unsigned long long s_thr;
  __shared__ int s_m;
  grid_dep_wait();
  grid_dep_launch();
  const int s = blockIdx.x, r = blockIdx.y, slices = gridDim.x;
  const int tid = threadIdx.x, lane = tid & 31;
  const InT* row = logits + logit_row<kDraftRows>(r, B) * ld;
  const int c0 = s * kSlice, c1 = min(V, c0 + kSlice);
  // element q of the thread: column c0 + kPer * (tid + 256 * (q / kPer)) + q % kPer
  auto col_of = [&](int q) { return c0 + kPer * (tid + kThreads * (q / kPer)) + q % kPer; };
  uint4 v[kQuads];
#pragma unroll
  for (int u = 0; u < kQuads; ++u) {
    const int c = c0 + kPer * (tid + kThreads * u);
    v[u] = c < c1 ? __ldcs(reinterpret_cast<const uint4*>(row + c)) : make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
  }
  // maximum of every 16-byte load (NaN skipped) and of the lane; a full
  // slice needs no column checks, a ragged one masks columns past c1
  const bool full = c1 - c0 == kSlice;
  float lm[kQuads];
#pragma unroll
  for (int u = 0; u < kQuads; ++u) lm[u] = load_max<InT>(v[u]);
  if (!full) {
#pragma unroll
    for (int u = 0; u < kQuads; ++u) {
      float m = -INFINITY;
#pragma unroll
      for (int e = 0; e < kPer; ++e)
        if (col_of(u * kPer + e) < c1) m = fmaxf(m, elem<InT>(v, u * kPer + e));
      lm[u] = m;
    }
  }
  float bv = -INFINITY;
#pragma unroll
  for (int u = 0; u < kQuads; ++u) bv = fmaxf(bv, lm[u]);
  uint32_t ob = ordered_bits(bv == 0.f ? 0.f : bv);
  // the warp's R-th largest lane maximum: remove the largest R - 1 times
  uint32_t rth = 0;
#pragma unroll
  for (int k = 0; k < R; ++k) {
    rth = __reduce_max_sync(0xffffffffu, ob);
    const int l = __ffs(__ballot_sync(0xffffffffu, ob == rth)) - 1;
    if (lane == l) ob = 0;
  }
  if (lane == 0) s_rw[tid >> 5] = rth;
  if (tid == 0) s_m = 0;
  __syncthreads();
  uint32_t tb = s_rw[0];
#pragma unroll
  for (int w = 1; w < kThreads / 32; ++w) tb = min(tb, s_rw[w]);
  // keys at or above thr: values at or above the bound (any column)
  unsigned long long thr = static_cast<unsigned long long>(tb) << 32;
  auto offer = [&](float x, int c) {
    if (c < c1 && x >= key_value(thr)) {   // k >= thr implies value(k) >= value(thr); NaN fails
      const unsigned long long k = logit_key(x, c);
      if (k >= thr) {
        const int at = atomicAdd(&s_m, 1);
        if (at < kCandCap) s_cand[at] = k;
      }
    }
  };
  const float tf0 = key_value(thr);
#pragma unroll
  for (int u = 0; u < kQuads; ++u) {
    if (lm[u] >= tf0) {   // rare: this load holds a value at or above the bound
#pragma unroll
      for (int e = 0; e < kPer; ++e) offer(elem<InT>(v, u * kPer + e), col_of(u * kPer + e));
    }
  }
  __syncthreads();
  while (s_m > kCandCap) {
    // ties overflowed the buffer: its K-th largest key is the next bound, and
    // the slice is read again from memory (the registers are no longer live)
    for (int j = tid; j < kCandCap; j += kThreads) {
      const unsigned long long k = s_cand[j];
      int rank = 0;
      for (int q = 0; q < kCandCap; ++q) rank += s_cand[q] > k;
      if (rank == K - 1) s_thr = k;
    }
    __syncthreads();
    thr = s_thr;
    if (tid == 0) s_m = 0;
    __syncthreads();
    for (int q = 0; q < kVals; ++q) {
      const int c = col_of(q);
      if (c < c1) {
        float x;
        if constexpr (In<InT>::kPerLoad == 4) x = row[c];
        else x = __uint_as_float(static_cast<uint32_t>(row[c]) << 16);
        offer(x, c);
      }
    }
    __syncthreads();
  }
  top_by_rank<K>(s_cand, s_m, tid, kThreads, part + (static_cast<size_t>(r) * slices + s) * K);
}

// Merge the slice lists of one row into its K largest keys, decreasing
// (zeros past the row's valid columns). Shared scratch: keys and kept hold
// slices * K entries each; s_thr and s_m are shared scalars. All nthr threads
// of the group call it; bar() synchronises the group.
template <int K, typename Bar>
__device__ __forceinline__ void merge_lists(const unsigned long long* __restrict__ src, int slices, int tid, int nthr,
                                            unsigned long long* keys, unsigned long long* kept,
                                            unsigned long long* s_thr, unsigned long long* s_lo, int* s_m,
                                            unsigned long long* out, Bar bar) {
  const int n = slices * K;
  constexpr int kMaxPer = 8;   // slices * K <= 8 * nthr
  unsigned long long kv[kMaxPer];
#pragma unroll
  for (int u = 0; u < kMaxPer; ++u) kv[u] = tid + nthr * u < n ? __ldcg(src + tid + nthr * u) : 0ull;
#pragma unroll
  for (int u = 0; u < kMaxPer; ++u)
    if (tid + nthr * u < n) keys[tid + nthr * u] = kv[u];
  if (tid == 0) {
    *s_thr = 0;
    s_lo[0] = ~0ull;
    *s_m = 0;
  }
  bar();
  // two lower bounds of the row's K-th largest key: the largest of the
  // slices' K-th keys, and, with c = ceil(K / slices) keys taken from every
  // slice (at least K in all), the smallest of the slices' c-th keys
  if (tid < slices) {
    const int c = (K + slices - 1) / slices;
    atomicMax(s_thr, keys[tid * K + K - 1]);
    atomicMin(s_lo, keys[tid * K + c - 1]);
  }
  bar();
  const unsigned long long t = max(*s_thr, s_lo[0]);
  for (int q = tid; q < n; q += nthr) {
    const unsigned long long k = keys[q];
    if (k != 0 && k >= t) kept[atomicAdd(s_m, 1)] = k;
  }
  bar();
  top_by_rank<K>(kept, *s_m, tid, nthr, out);
  bar();
}

}  // namespace topk
}  // namespace dfl
