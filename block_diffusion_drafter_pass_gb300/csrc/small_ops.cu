// small_ops.cu - row-wise and per-sequence kernels of the drafter pass:
// block embedding + input RMSNorm, RMSNorm, greedy verify + commit (warp
// ballot), the position advance after a context append, and the bf16 row
// argmax that turns target logits into the target's greedy ids.
#include <cuda.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

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

// Block rows [anchor, MASK x (B-1)] per sequence -> fp32 residual x and the
// first layer's normalised input h (bf16).
__global__ void __launch_bounds__(kRowThreads) embed_norm_kernel(const uint16_t* __restrict__ embed,
                                                                 const int32_t* __restrict__ anchors, int mask_id,
                                                                 int vocab, const __grid_constant__ SeqMeta meta,
                                                                 int H, const uint16_t* __restrict__ gain, float eps,
                                                                 float* __restrict__ x, uint16_t* __restrict__ h,
                                                                 int* status) {
  __shared__ float red[32];
  grid_dep_wait();
  const int m = blockIdx.x;
  const int i = m / meta.B, j = m - i * meta.B;
  int id = j == 0 ? anchors[i] : mask_id;
  if (id < 0 || id >= vocab) {
    if (threadIdx.x == 0) latch_status(status, kDevBounds);
    id = 0;
  }
  const uint16_t* e = embed + static_cast<size_t>(id) * H;
  float* xr = x + static_cast<size_t>(m) * H;
  float ss = 0.f;
  for (int c = threadIdx.x; c < H; c += blockDim.x) {
    const float v = bf16_to_f32(e[c]);
    xr[c] = v;
    ss += v * v;
  }
  const float inv = rsqrtf(block_sum(ss, red) / H + eps);
  for (int c = threadIdx.x; c < H; c += blockDim.x)
    h[static_cast<size_t>(m) * H + c] = f32_to_bf16(xr[c] * inv * bf16_to_f32(gain[c]));
  grid_dep_launch();
}

// out[row'] = x[row] / sqrt(mean(x^2) + eps) * gain. With skip_B > 0 the
// first row of every group of skip_B rows is dropped (rows j >= 1 of each
// block are compacted to [n_seq*(B-1)]).
__global__ void __launch_bounds__(kRowThreads) rmsnorm_kernel(const float* __restrict__ x, int H,
                                                              const uint16_t* __restrict__ gain, float eps,
                                                              uint16_t* __restrict__ out, int skip_B) {
  __shared__ float red[32];
  grid_dep_wait();
  int m = blockIdx.x, mo = m;
  if (skip_B > 0) {
    const int i = m / (skip_B - 1), j = m - i * (skip_B - 1);
    m = i * skip_B + j + 1;
    mo = blockIdx.x;
  }
  const float* xr = x + static_cast<size_t>(m) * H;
  float ss = 0.f;
  for (int c = threadIdx.x; c < H; c += blockDim.x) {
    const float v = xr[c];
    ss += v * v;
  }
  const float inv = rsqrtf(block_sum(ss, red) / H + eps);
  for (int c = threadIdx.x; c < H; c += blockDim.x)
    out[static_cast<size_t>(mo) * H + c] = f32_to_bf16(xr[c] * inv * bf16_to_f32(gain[c]));
  grid_dep_launch();
}

// One warp per sequence: lane j flags draft[j] != target[j]; the first set
// bit of the ballot is the first mismatch a; tau = a + 1, bonus = target[a].
// Then commit min(tau, pending) pending tokens and drop the rest.
__global__ void verify_kernel(const __grid_constant__ SeqMeta meta, SeqState st, const int32_t* __restrict__ drafts,
                              const int32_t* __restrict__ targets, int32_t* __restrict__ tau,
                              int32_t* __restrict__ bonus) {
  grid_dep_wait();
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
  const int i = threadIdx.x;
  if (i >= meta.n_seq) return;
  const int n = meta.row0[i + 1] - meta.row0[i];
  const int slot = meta.slot[i];
  if (pending) st.pend[slot] += n;
  else st.len[slot] += n;
}

// Row argmax of bf16 logits, lowest index on ties: the per-thread best is kept
// as a 64-bit key (ordered value << 32 | ~index) so one max picks both.
__global__ void __launch_bounds__(kRowThreads) rows_argmax_bf16_kernel(const uint16_t* __restrict__ logits, int cols,
                                                                       int32_t* __restrict__ out, int vec_ok) {
  __shared__ unsigned long long red[32];
  const int row = blockIdx.x;
  const uint16_t* p = logits + static_cast<size_t>(row) * cols;
  unsigned long long best = 0ull;
  auto consider = [&](float v, int idx) {
    const unsigned long long k =
        (static_cast<unsigned long long>(ordered_key(v)) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(idx));
    best = k > best ? k : best;
  };
  if (vec_ok) {
    const int nvec = cols >> 3;
    const uint4* pv = reinterpret_cast<const uint4*>(p);
    int vi = threadIdx.x;
    for (; vi + 3 * kRowThreads < nvec; vi += 4 * kRowThreads) {
      uint4 w[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) w[u] = __ldcs(pv + vi + u * kRowThreads);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t ws[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
        const int base = (vi + u * kRowThreads) * 8;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          consider(__uint_as_float(ws[q] << 16), base + 2 * q);
          consider(__uint_as_float(ws[q] & 0xFFFF0000u), base + 2 * q + 1);
        }
      }
    }
    for (; vi < nvec; vi += kRowThreads) {
      const uint4 w = __ldcs(pv + vi);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        consider(__uint_as_float(ws[q] << 16), vi * 8 + 2 * q);
        consider(__uint_as_float(ws[q] & 0xFFFF0000u), vi * 8 + 2 * q + 1);
      }
    }
    for (int c = (nvec << 3) + threadIdx.x; c < cols; c += kRowThreads) consider(bf16_to_f32(p[c]), c);
  } else {
    for (int c = threadIdx.x; c < cols; c += kRowThreads) consider(bf16_to_f32(p[c]), c);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long t = __shfl_xor_sync(0xffffffffu, best, o);
    best = t > best ? t : best;
  }
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = best;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kRowThreads / 32; ++w) best = red[w] > best ? red[w] : best;
    out[row] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(best & 0xFFFFFFFFull));
  }
}

}  // namespace

cudaError_t launch_embed_norm(const uint16_t* embed, const int32_t* anchors, int mask_id, int vocab,
                              const SeqMeta& meta, int H, const uint16_t* gain, float eps, float* x, uint16_t* h,
                              int* status, cudaStream_t s) {
  const int rows = meta.n_seq * meta.B;
  if (rows == 0) return cudaSuccess;
  embed_norm_kernel<<<rows, kRowThreads, 0, s>>>(embed, anchors, mask_id, vocab, meta, H, gain, eps, x, h, status);
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm(const float* x, int rows, int H, const uint16_t* gain, float eps, uint16_t* out, int skip_B,
                           cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  rmsnorm_kernel<<<rows, kRowThreads, 0, s>>>(x, H, gain, eps, out, skip_B);
  return cudaGetLastError();
}

cudaError_t launch_verify(const SeqMeta& meta, SeqState st, const int32_t* drafts, const int32_t* targets,
                          int32_t* tau, int32_t* bonus, cudaStream_t s) {
  if (meta.n_seq == 0) return cudaSuccess;
  const int warps = 4;
  verify_kernel<<<(meta.n_seq + warps - 1) / warps, warps * 32, 0, s>>>(meta, st, drafts, targets, tau, bonus);
  return cudaGetLastError();
}

cudaError_t launch_fuse_advance(const SeqMeta& meta, SeqState st, int pending, cudaStream_t s) {
  if (meta.n_seq == 0) return cudaSuccess;
  fuse_advance_kernel<<<1, kMaxBatch, 0, s>>>(meta, st, pending);
  return cudaGetLastError();
}

cudaError_t launch_rows_argmax_bf16(const uint16_t* logits, int rows, int cols, int32_t* out, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  const int vec_ok = (cols % 8 == 0) && (reinterpret_cast<uintptr_t>(logits) % 16 == 0);
  rows_argmax_bf16_kernel<<<rows, kRowThreads, 0, s>>>(logits, cols, out, vec_ok);
  return cudaGetLastError();
}

}  // namespace dfl
