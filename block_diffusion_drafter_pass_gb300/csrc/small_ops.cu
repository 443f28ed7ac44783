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

// Block rows [anchor, MASK x (B-1)] per sequence (drafter), or the caller's
// block ids (target pass: ids[m] for row m) -> fp32 residual x, the first
// layer's RMSNorm input bf16(x * gain) and sum(x^2) per row (the GEMM that
// consumes the row applies 1/sqrt(mean + eps)). One CTA per row, 16-byte
// loads of the bf16 embedding row.
__global__ void __launch_bounds__(kRowThreads) embed_kernel(const uint16_t* __restrict__ embed,
                                                            const int32_t* __restrict__ anchors, int mask_id,
                                                            const int32_t* __restrict__ ids, int vocab,
                                                            const __grid_constant__ SeqMeta meta, int H,
                                                            const uint16_t* __restrict__ gain, float* __restrict__ x,
                                                            uint16_t* __restrict__ hg, float* __restrict__ ss,
                                                            int* status) {
  __shared__ float red[32];
  grid_dep_wait();
  grid_dep_launch();
  const int m = blockIdx.x;
  const int i = m / meta.B, j = m - i * meta.B;
  int id = ids ? ids[m] : (j == 0 ? anchors[i] : mask_id);
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

// A wait that nothing satisfies: one thread waits on an mbarrier no thread
// arrives on, gives up after limit_ns and latches the timeout bit, the path
// every bounded wait of the library takes when it runs out.
__global__ void wait_probe_kernel(unsigned long long limit_ns, int* status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_mbar_init();
  if (!mbar_wait_for(&bar, 0, limit_ns)) latch_status(status, kDevTimeout);
}

// Target pass: the block's keys (rotated) and values of one layer, from the
// projection's block buffers (keys [row][n_kv][d], values transposed
// [sequence][n_kv][d][64 slots]), appended to the paged pool at positions
// len + j, the slots after the sequence's committed tokens. One CTA per block
// row.
__global__ void block_kv_append_kernel(const __grid_constant__ SeqMeta meta, SeqState st, int layer,
                                       const uint16_t* __restrict__ kb, const uint16_t* __restrict__ vb,
                                       uint16_t* __restrict__ pool, int pool_pages, int n_kv, int d, int* status) {
  grid_dep_wait();
  grid_dep_launch();
  const int m = blockIdx.x;
  const int i = m / meta.B, j = m - i * meta.B;
  const int slot = meta.slot[i];
  const int pos = st.len[slot] + j;
  const int pi = pos / kPage, s64 = pos - pi * kPage;
  const int page = pi < st.pages_per_seq ? st.page_table[static_cast<size_t>(slot) * st.pages_per_seq + pi] : -1;
  if (page < 0 || page >= pool_pages) {
    if (threadIdx.x == 0) latch_status(status, kDevBounds);
    return;
  }
  const size_t base = (static_cast<size_t>(layer) * pool_pages + page) * 2 * n_kv * kPage * d;
  for (int e = threadIdx.x; e < n_kv * d; e += blockDim.x) {
    const int h = e / d, di = e - h * d;
    pool[base + (static_cast<size_t>(h) * kPage + s64) * d + di] = kb[(static_cast<size_t>(m) * n_kv + h) * d + di];
    pool[base + static_cast<size_t>(n_kv) * kPage * d + (static_cast<size_t>(h) * d + di) * kPage + s64] =
        vb[((static_cast<size_t>(i) * n_kv + h) * d + di) * kPage + j];
  }
}

// Target pass: the residual stream after a feature layer, x [M][H] fp32, to
// columns col0 .. col0+H-1 of the feature rows feats [M][ld] bf16.
__global__ void feat_copy_kernel(const float* __restrict__ x, int H, uint16_t* __restrict__ feats, int ld, int col0) {
  grid_dep_wait();
  grid_dep_launch();
  const int m = blockIdx.x;
  const float4* xr = reinterpret_cast<const float4*>(x + static_cast<size_t>(m) * H);
  uint2* fr = reinterpret_cast<uint2*>(feats + static_cast<size_t>(m) * ld + col0);
  for (int c = threadIdx.x; c < H / 4; c += blockDim.x) {
    const float4 v = xr[c];
    fr[c] = make_uint2(static_cast<uint32_t>(f32_to_bf16(v.x)) | (static_cast<uint32_t>(f32_to_bf16(v.y)) << 16),
                       static_cast<uint32_t>(f32_to_bf16(v.z)) | (static_cast<uint32_t>(f32_to_bf16(v.w)) << 16));
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
//
// Each CTA reduces one segment of one row. A row is split over a cluster of
// KC CTAs (KC = 1 when there are enough rows to fill the GPU); their partial
// keys meet in the first CTA's shared memory (distributed shared memory), so
// no global scratch is needed. When rows are 16-byte aligned (cols % 8 == 0)
// the segment streams through a ring of kAmStages bulk copies of kAmChunk
// columns, so a CTA keeps 64 KB in flight with few registers and the GPU's
// CTA scheduler balances whole rows over the SMs; otherwise threads read the
// segment directly.
constexpr int kAmThreads = 512;
constexpr int kAmWarps = kAmThreads / 32;
constexpr int kAmChunk = 8192;   // columns per ring stage (16 KB)
constexpr int kAmStages = 4;

__device__ __forceinline__ unsigned long long argmax_key(float v, int idx) {
  return (static_cast<unsigned long long>(ordered_key(v)) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(idx));
}

__device__ __forceinline__ unsigned long long max_key(unsigned long long a, unsigned long long b) {
  return a > b ? a : b;
}

// Key of a (value, column) candidate: larger values first, then lower
// columns; -0 and +0 are one value (as a float comparison sees them).
__device__ __forceinline__ unsigned long long cand_key(float v, int idx) {
  return idx < 0 ? 0ull : argmax_key(v == 0.f ? 0.f : v, idx);
}

template <int KC>
__global__ void __launch_bounds__(kAmThreads)
    rows_argmax_bf16_kernel(const uint16_t* __restrict__ logits, int cols, int32_t* __restrict__ out, int* status,
                            int ring) {
  extern __shared__ __align__(128) uint8_t am_ring[];   // kAmStages x kAmChunk bf16 (ring mode)
  __shared__ __align__(8) uint64_t full[kAmStages], empty[kAmStages];
  __shared__ unsigned long long red[kAmWarps];
  __shared__ unsigned long long cta_best;
  __shared__ volatile int abort_flag;
  const int seg = static_cast<int>(blockIdx.x % KC), row = static_cast<int>(blockIdx.x / KC);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int per = ((cols + KC * 8 - 1) / (KC * 8)) * 8;   // multiple of 8 columns
  const int c_lo = min(cols, seg * per), c_hi = min(cols, c_lo + per);
  const uint16_t* p = logits + static_cast<size_t>(row) * cols;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kAmStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kAmWarps);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  grid_dep_launch();   // dependents read the result only after their own wait
  grid_dep_wait();
  unsigned long long b = 0ull;
  if (ring) {
    // This thread's running (value, first column): a vector's maximum comes
    // from packed bf16 pairs, and only a vector that beats the running value
    // is searched for the first column holding its maximum.
    float bv = -INFINITY;
    int bi = -1;
    const int n = (c_hi - c_lo + kAmChunk - 1) / kAmChunk;   // chunks of this segment
    auto issue = [&](int k) {
      const int s = k % kAmStages;
      const int c0 = c_lo + k * kAmChunk, len = min(kAmChunk, c_hi - c0);
      mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(len) * 2u);
      bulk_load(am_ring + static_cast<size_t>(s) * kAmChunk * 2, p + c0, static_cast<uint32_t>(len) * 2u, &full[s]);
    };
    int issued = 0;   // thread 0's count of copies issued
    if (threadIdx.x == 0)
      for (; issued < n && issued < kAmStages; ++issued) issue(issued);
    for (int k = 0; k < n; ++k) {
      const int s = k % kAmStages;
      if (!mbar_wait(&full[s], (k / kAmStages) & 1, &abort_flag)) {
        abort_flag = 1;
        latch_status(status, kDevTimeout);
        break;
      }
      const int c0 = c_lo + k * kAmChunk, len = min(kAmChunk, c_hi - c0);
      const uint4* sv = reinterpret_cast<const uint4*>(am_ring + static_cast<size_t>(s) * kAmChunk * 2);
      for (int v = threadIdx.x; v < (len >> 3); v += kAmThreads) {
        const uint4 w = sv[v];
        const __nv_bfloat162 m2 =
            __hmax2(__hmax2(*reinterpret_cast<const __nv_bfloat162*>(&w.x), *reinterpret_cast<const __nv_bfloat162*>(&w.y)),
                    __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&w.z), *reinterpret_cast<const __nv_bfloat162*>(&w.w)));
        const float m = fmaxf(__low2float(m2), __high2float(m2));
        if (m > bv || bi < 0) {
          const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
          int q = 0;
          for (; q < 8; ++q) {
            const uint32_t h = (q & 1) ? (ws[q >> 1] & 0xFFFF0000u) : (ws[q >> 1] << 16);
            if (__uint_as_float(h) == m) break;
          }
          bi = c0 + v * 8 + (q < 8 ? q : 0);
          bv = m;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      if (threadIdx.x == 0 && k + kAmStages < n) {
        // every warp has read this stage: refill it
        if (!mbar_wait(&empty[s], (k / kAmStages) & 1, &abort_flag)) {
          abort_flag = 1;
          latch_status(status, kDevTimeout);
        } else {
          issue(k + kAmStages);
          ++issued;
        }
      }
    }
    b = cand_key(bv, bi);
    if (threadIdx.x == 0 && abort_flag) {
      // copies still in flight land before shared memory is released
      for (int k = max(0, issued - kAmStages); k < issued; ++k) mbar_wait(&full[k % kAmStages], (k / kAmStages) & 1);
    }
  } else {
    float bv = -INFINITY;
    int bi = -1;
    for (int c = c_lo + threadIdx.x; c < c_hi; c += kAmThreads) {
      const float v = bf16_to_f32(p[c]);
      if (v > bv || bi < 0) {
        bv = v;
        bi = c;
      }
    }
    b = cand_key(bv, bi);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) b = max_key(b, __shfl_xor_sync(0xffffffffu, b, o));
  if (lane == 0) red[warp] = b;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kAmWarps; ++w) b = max_key(b, red[w]);
    cta_best = abort_flag ? 0xFFFFFFFF00000000ull : b;   // a segment that gave up marks the row: id -1
  }
  if constexpr (KC == 1) {
    if (threadIdx.x == 0)
      out[row] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(cta_best & 0xFFFFFFFFull));
  } else {
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    if (seg == 0 && threadIdx.x == 0) {
      unsigned long long k = 0ull;
      for (int r = 0; r < KC; ++r) k = max_key(k, *cluster.map_shared_rank(&cta_best, r));
      out[row] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(k & 0xFFFFFFFFull));
    }
    cluster.sync();   // keep every CTA's shared memory alive until the first one has read it
  }
}

template <int KC>
cudaError_t launch_argmax_kc(const uint16_t* logits, int rows, int cols, int32_t* out, int* status, int ring,
                             cudaStream_t s) {
  const size_t smem = ring ? static_cast<size_t>(kAmStages) * kAmChunk * 2 : 0;
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(rows_argmax_bf16_kernel<KC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(kAmStages * kAmChunk * 2));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  if constexpr (KC == 1)
    return launch_pdl(rows_argmax_bf16_kernel<KC>, dim3(rows), dim3(kAmThreads), smem, s, logits, cols, out, status,
                      ring);
  else
    return launch_pdl_cluster(rows_argmax_bf16_kernel<KC>, dim3(rows * KC), dim3(kAmThreads), smem, KC, s, logits,
                              cols, out, status, ring);
}

}  // namespace

cudaError_t launch_embed(const uint16_t* embed, const int32_t* anchors, int mask_id, const int32_t* ids, int vocab,
                         const SeqMeta& meta, int H, const uint16_t* gain, float* x, uint16_t* hg, float* ss,
                         int* status, cudaStream_t s) {
  const int rows = meta.n_seq * meta.B;
  if (rows == 0) return cudaSuccess;
  return launch_pdl(embed_kernel, dim3(rows), dim3(kRowThreads), 0, s, embed, anchors, mask_id, ids, vocab, meta, H,
                    gain, x, hg, ss, status);
}

cudaError_t launch_block_kv_append(const SeqMeta& meta, SeqState st, int layer, const uint16_t* kb, const uint16_t* vb,
                                   uint16_t* pool, int pool_pages, int n_kv, int d, int* status, cudaStream_t s) {
  const int rows = meta.n_seq * meta.B;
  if (rows == 0) return cudaSuccess;
  return launch_pdl(block_kv_append_kernel, dim3(rows), dim3(256), 0, s, meta, st, layer, kb, vb, pool, pool_pages,
                    n_kv, d, status);
}

cudaError_t launch_feat_copy(const float* x, int M, int H, uint16_t* feats, int ld, int col0, cudaStream_t s) {
  if (M == 0) return cudaSuccess;
  return launch_pdl(feat_copy_kernel, dim3(M), dim3(256), 0, s, x, H, feats, ld, col0);
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

cudaError_t launch_wait_probe(unsigned long long limit_ns, int* status, cudaStream_t s) {
  wait_probe_kernel<<<1, 32, 0, s>>>(limit_ns, status);
  return cudaGetLastError();
}

cudaError_t launch_page_updates(const PageUpdates& u, int* table, cudaStream_t s) {
  if (u.n <= 0) return cudaSuccess;
  return launch_pdl(page_table_update_kernel, dim3(1), dim3(256), 0, s, u, table);
}

cudaError_t launch_rows_argmax_bf16(const uint16_t* logits, int rows, int cols, int32_t* out, cudaStream_t s) {
  int* status = nullptr;   // no context: a row whose wait gave up reads -1 instead
  if (rows == 0) return cudaSuccess;
  const int ring = (cols % 8 == 0) && (reinterpret_cast<uintptr_t>(logits) % 16 == 0);
  // CTAs per row: enough CTAs to cover the SMs a few times over
  if (rows >= 256) return launch_argmax_kc<1>(logits, rows, cols, out, status, ring, s);
  if (rows >= 128) return launch_argmax_kc<2>(logits, rows, cols, out, status, ring, s);
  if (rows >= 64) return launch_argmax_kc<4>(logits, rows, cols, out, status, ring, s);
  return launch_argmax_kc<8>(logits, rows, cols, out, status, ring, s);
}

}  // namespace dfl
