// small_ops.cu - row-wise and per-sequence kernels of the drafter pass:
// block embedding (with the first layer's folded RMSNorm inputs), greedy
// verify + commit (warp ballot), the position advance after a context append,
// and the bf16 row argmax that turns target logits into the target's greedy ids.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cooperative_groups.h>

#include "internal.h"
#include "ptx.cuh"

namespace cg = cooperative_groups;

namespace dfl {
namespace {

constexpr int kRowThreads = 256;

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) red[w] = v;
  __syncthreads();
  float t = 0.f;
  if (threadIdx.x < 32) {
    t = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if (threadIdx.x == 0) red[0] = t;
  }
  __syncthreads();
  const float r = red[0];
  __syncthreads();
  return r;
}

// Block rows [anchor, MASK x (B-1)] per sequence -> fp32 residual x, the
// first layer's RMSNorm input bf16(x * gain) and sum(x^2) per row (the GEMM
// that consumes the row applies 1/sqrt(mean + eps)). One CTA per row,
// 16-byte loads of the bf16 embedding row.
__global__ void __launch_bounds__(kRowThreads) embed_kernel(const uint16_t* __restrict__ embed,
                                                            const int32_t* __restrict__ anchors, int mask_id,
                                                            int vocab, const __grid_constant__ SeqMeta meta, int H,
                                                            const uint16_t* __restrict__ gain, float* __restrict__ x,
                                                            uint16_t* __restrict__ hg, float* __restrict__ ss,
                                                            int* status) {
  __shared__ float red[32];
  grid_dep_wait();
  grid_dep_launch();
  const int m = blockIdx.x;
  const int i = m / meta.B, j = m - i * meta.B;
  int id = j == 0 ? anchors[i] : mask_id;
  if (id < 0 || id >= vocab) {
    if (threadIdx.x == 0) latch_status(status, kDevBounds);
    id = 0;
  }
  const uint4* e = reinterpret_cast<const uint4*>(embed + static_cast<size_t>(id) * H);
  const uint4* gv = reinterpret_cast<const uint4*>(gain);
  float4* xr = reinterpret_cast<float4*>(x + static_cast<size_t>(m) * H);
  uint4* hr = reinterpret_cast<uint4*>(hg + static_cast<size_t>(m) * H);
  float acc = 0.f;
  for (int c = threadIdx.x; c < H / 8; c += blockDim.x) {
    const uint4 w = e[c], g = gv[c];
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w}, gs[4] = {g.x, g.y, g.z, g.w};
    float f[8];
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      f[2 * q] = __uint_as_float(ws[q] << 16);
      f[2 * q + 1] = __uint_as_float(ws[q] & 0xFFFF0000u);
      const float g0 = __uint_as_float(gs[q] << 16), g1 = __uint_as_float(gs[q] & 0xFFFF0000u);
      o[q] = static_cast<uint32_t>(f32_to_bf16(f[2 * q] * g0)) |
             (static_cast<uint32_t>(f32_to_bf16(f[2 * q + 1] * g1)) << 16);
      acc += f[2 * q] * f[2 * q] + f[2 * q + 1] * f[2 * q + 1];
    }
    xr[2 * c] = make_float4(f[0], f[1], f[2], f[3]);
    xr[2 * c + 1] = make_float4(f[4], f[5], f[6], f[7]);
    hr[c] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  const float tot = block_sum(acc, red);
  if (threadIdx.x == 0) ss[m] = tot;
}

// One warp per sequence: lane j flags draft[j] != target[j]; the first set
// bit of the ballot is the first mismatch a; tau = a + 1, bonus = target[a].
// Then commit min(tau, pending) pending tokens and drop the rest.
__global__ void verify_kernel(const __grid_constant__ SeqMeta meta, SeqState st, const int32_t* __restrict__ drafts,
                              const int32_t* __restrict__ targets, int32_t* __restrict__ tau,
                              int32_t* __restrict__ bonus) {
  grid_dep_wait();
  grid_dep_launch();
  const int i = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (i >= meta.n_seq) return;
  const int B = meta.B;
  const bool mismatch =
      lane < B - 1 && drafts[static_cast<size_t>(i) * (B - 1) + lane] != targets[static_cast<size_t>(i) * B + lane];
  const uint32_t mm = __ballot_sync(0xffffffffu, mismatch);
  const int a = mm ? (__ffs(mm) - 1) : (B - 1);
  if (lane == 0) {
    tau[i] = a + 1;
    bonus[i] = targets[static_cast<size_t>(i) * B + a];
    const int slot = meta.slot[i];
    const int p = st.pend[slot];
    st.len[slot] += min(a + 1, p);
    st.pend[slot] = 0;
  }
}

__global__ void fuse_advance_kernel(const __grid_constant__ SeqMeta meta, SeqState st, int pending) {
  grid_dep_wait();
  grid_dep_launch();
  const int i = threadIdx.x;
  if (i >= meta.n_seq) return;
  const int n = meta.row0[i + 1] - meta.row0[i];
  const int slot = meta.slot[i];
  if (pending) st.pend[slot] += n;
  else st.len[slot] += n;
}

// Dependents may start at once (none reads the page table before its own
// wait; the attention kernel's early reads sit behind the draft's embedding
// kernel). The entries are written after the wait, when every earlier reader
// of the table has completed.
__global__ void page_table_update_kernel(const __grid_constant__ PageUpdates u, int* table) {
  grid_dep_launch();
  grid_dep_wait();
  for (int k = threadIdx.x; k < u.n; k += blockDim.x) table[u.idx[k]] = u.page[k];
}

// Row argmax of bf16 logits, lowest index on ties: the per-thread best is kept
// as a 64-bit key (ordered value << 32 | ~index) so one max picks both.
// Each row is split over a cluster of kArgCluster CTAs; their partial keys
// meet in the first CTA's shared memory (distributed shared memory), so no
// global scratch is needed.
constexpr int kArgCluster = 8;
constexpr int kArgThreads = 512;

__device__ __forceinline__ unsigned long long argmax_key(float v, int idx) {
  return (static_cast<unsigned long long>(ordered_key(v)) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(idx));
}

__global__ void __cluster_dims__(1, kArgCluster, 1) __launch_bounds__(kArgThreads)
    rows_argmax_bf16_kernel(const uint16_t* __restrict__ logits, int cols, int32_t* __restrict__ out, int vec_ok) {
  __shared__ unsigned long long red[kArgThreads / 32];
  __shared__ unsigned long long cta_best;
  cg::cluster_group cluster = cg::this_cluster();
  grid_dep_wait();
  grid_dep_launch();
  const int row = blockIdx.x;
  const int seg = static_cast<int>(cluster.block_rank());
  const int per = ((cols + kArgCluster * 8 - 1) / (kArgCluster * 8)) * 8;   // multiple of 8 columns
  const int c_lo = min(cols, seg * per), c_hi = min(cols, c_lo + per);
  const uint16_t* p = logits + static_cast<size_t>(row) * cols;
  unsigned long long best = 0ull;
  if (vec_ok) {
    const uint4* pv = reinterpret_cast<const uint4*>(p + c_lo);
    const int nvec = (c_hi - c_lo) >> 3;
    int vi = threadIdx.x;
    for (; vi + 3 * kArgThreads < nvec; vi += 4 * kArgThreads) {
      uint4 w[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) w[u] = __ldcs(pv + vi + u * kArgThreads);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t ws[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
        const int base = c_lo + (vi + u * kArgThreads) * 8;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const unsigned long long k0 = argmax_key(__uint_as_float(ws[q] << 16), base + 2 * q);
          const unsigned long long k1 = argmax_key(__uint_as_float(ws[q] & 0xFFFF0000u), base + 2 * q + 1);
          best = k0 > best ? k0 : best;
          best = k1 > best ? k1 : best;
        }
      }
    }
    for (; vi < nvec; vi += kArgThreads) {
      const uint4 w = __ldcs(pv + vi);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const unsigned long long k0 = argmax_key(__uint_as_float(ws[q] << 16), c_lo + vi * 8 + 2 * q);
        const unsigned long long k1 = argmax_key(__uint_as_float(ws[q] & 0xFFFF0000u), c_lo + vi * 8 + 2 * q + 1);
        best = k0 > best ? k0 : best;
        best = k1 > best ? k1 : best;
      }
    }
    for (int c = c_lo + (nvec << 3) + threadIdx.x; c < c_hi; c += kArgThreads) {
      const unsigned long long k = argmax_key(bf16_to_f32(p[c]), c);
      best = k > best ? k : best;
    }
  } else {
    for (int c = c_lo + threadIdx.x; c < c_hi; c += kArgThreads) {
      const unsigned long long k = argmax_key(bf16_to_f32(p[c]), c);
      best = k > best ? k : best;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long t = __shfl_xor_sync(0xffffffffu, best, o);
    best = t > best ? t : best;
  }
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = best;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kArgThreads / 32; ++w) best = red[w] > best ? red[w] : best;
    cta_best = best;
  }
  cluster.sync();
  if (seg == 0 && threadIdx.x == 0) {
    unsigned long long b = 0ull;
    for (int r = 0; r < kArgCluster; ++r) {
      const unsigned long long k = *cluster.map_shared_rank(&cta_best, r);
      b = k > b ? k : b;
    }
    out[row] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(b & 0xFFFFFFFFull));
  }
  cluster.sync();   // keep every CTA's shared memory alive until the first one has read it
}

}  // namespace

cudaError_t launch_embed(const uint16_t* embed, const int32_t* anchors, int mask_id, int vocab, const SeqMeta& meta,
                         int H, const uint16_t* gain, float* x, uint16_t* hg, float* ss, int* status, cudaStream_t s) {
  const int rows = meta.n_seq * meta.B;
  if (rows == 0) return cudaSuccess;
  return launch_pdl(embed_kernel, dim3(rows), dim3(kRowThreads), 0, s, embed, anchors, mask_id, vocab, meta, H, gain,
                    x, hg, ss, status);
}

cudaError_t launch_verify(const SeqMeta& meta, SeqState st, const int32_t* drafts, const int32_t* targets,
                          int32_t* tau, int32_t* bonus, cudaStream_t s) {
  if (meta.n_seq == 0) return cudaSuccess;
  const int warps = 4;
  return launch_pdl(verify_kernel, dim3((meta.n_seq + warps - 1) / warps), dim3(warps * 32), 0, s, meta, st, drafts,
                    targets, tau, bonus);
}

cudaError_t launch_fuse_advance(const SeqMeta& meta, SeqState st, int pending, cudaStream_t s) {
  if (meta.n_seq == 0) return cudaSuccess;
  return launch_pdl(fuse_advance_kernel, dim3(1), dim3(kMaxBatch), 0, s, meta, st, pending);
}

cudaError_t launch_page_updates(const PageUpdates& u, int* table, cudaStream_t s) {
  if (u.n <= 0) return cudaSuccess;
  return launch_pdl(page_table_update_kernel, dim3(1), dim3(256), 0, s, u, table);
}

cudaError_t launch_rows_argmax_bf16(const uint16_t* logits, int rows, int cols, int32_t* out, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  const int vec_ok = (cols % 8 == 0) && (reinterpret_cast<uintptr_t>(logits) % 16 == 0);
  return launch_pdl(rows_argmax_bf16_kernel, dim3(rows, kArgCluster), dim3(kArgThreads), 0, s, logits, cols, out,
                    vec_ok);
}

}  // namespace dfl
