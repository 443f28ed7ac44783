// conv.cu - the two-tap dynamic convolution of the DFlash 2 drafter ("DFlash 2"
// notes, "Solution - Two-Tap Dynamic Convolution"): around each attention and
// feed-forward sublayer, over the block positions of each sequence,
//   Conv(x)_t = k_{t,0} * x_t + k_{t,1} * x_{t-1}      (* elementwise, x_{-1} = 0)
// with coefficients k_{t,i} = base_i + U_i (V_i x_t), a rank-r correction
// computed from the position's own input.
//
// One apply kernel per convolution site. A CTA takes 32 columns and 16 rows
// (128 CTAs per 16 rows at hidden 4096, so a batch-1 block spreads over the
// GPU); its slices of U and of the next site's V^T arrive by bulk copies
// issued before the wait on the previous kernel (the pass never writes
// weights). It forms the rank-r products U_i P_t (P_t = V x_t, 2r values per
// row, made before: by the GEMM that produced the site's input, or by the
// previous apply kernel), the two-tap combination and then either
//   input sites  (before a sublayer): bf16 Conv(RMSNorm(x)) -> the sublayer's
//                GEMM input, RMSNorm(x) from the fp32 residual stream;
//   output sites (after a sublayer):  x += Conv(y); bf16(x * g) and the row's
//                sum of x^2 over the 32 columns (the next RMSNorm's parts);
//                and the next input site's products V_next (x * g) over these
//                columns, added into an fp32 accumulator (the input site
//                applies the row's RMSNorm scale; it also zeroes the other
//                accumulator for the output site after it).
// The per-CTA products (16 rows x 32 columns x r for U P, 16 x 2r x 32 for
// V (x g)) run on the tensor cores as warp-level tf32 products with fp32
// sums: operands straight from the bf16 weight slices (exact in tf32) and
// the fp32 rows rounded to tf32.
#include <cuda.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace dfl {
namespace {

constexpr int kCols = kConvCols;   // columns per CTA
constexpr int kRows = 16;          // rows per CTA
constexpr int kThreads = 512;      // one thread per (column, row); 16 warps hide the loads' latency

// RMSNorm scales of rows m_first .. m_first + n - 1 (n <= 17) into sc[], by
// the whole block: eight threads per row, thread q adding parts q, q + 8, ...
// (loads issued together), then the eight sums in a fixed tree - the sum
// order and formula of the GEMM's consumer side. Rows outside [0, M) get 0.
// Ends with a barrier.
__device__ __forceinline__ void rms_scales(const float* ss, int parts, int ld, int m_first, int n, int M,
                                           float inv_hidden, float eps, float* part_sums, float* sc) {
  for (int i = threadIdx.x; i < n * 8; i += kThreads) {
    const int row = i >> 3, q = i & 7, m = m_first + row;
    float acc = 0.f;
    if (m >= 0 && m < M) {
      float v[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const int p = q + 8 * k;
        v[k] = p < parts ? __ldcg(ss + static_cast<size_t>(p) * ld + m) : 0.f;
      }
#pragma unroll
      for (int k = 0; k < 16; ++k) acc += v[k];
      for (int p = q + 128; p < parts; p += 8) acc += __ldcg(ss + static_cast<size_t>(p) * ld + m);
    }
    part_sums[i] = acc;
  }
  __syncthreads();
  if (threadIdx.x < n) {
    const float* a = part_sums + threadIdx.x * 8;
    const float s = ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]));
    const int mm = m_first + static_cast<int>(threadIdx.x);
    sc[threadIdx.x] = mm >= 0 && mm < M ? rsqrtf(s * inv_hidden + eps) : 0.f;
  }
  __syncthreads();
}

__device__ __forceinline__ uint32_t to_tf32(float f) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(f));
  return r;
}

// D (16 x 8, fp32) += A (16 x 8, tf32, row-major) * B (8 x 8, tf32, by
// column): the warp-level tensor-core product. Fragments (g = lane / 4,
// q = lane % 4): a0 (g, q), a1 (g + 8, q), a2 (g, q + 4), a3 (g + 8, q + 4);
// b0 (k q, n g), b1 (k q + 4, n g); d0/d1 (g, 2q / 2q + 1), d2/d3 (g + 8, ...).
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t bf16_bits_f32(uint16_t b) { return static_cast<uint32_t>(b) << 16; }

struct ConvLayout {
  int u, vt, p, x, hq, kt, base, sc, scp, total;
  int p_ld;   // row pitch of p (2r + 4 words: the fragment loads of 8 rows cover distinct banks)
};

constexpr int kHqLd = kCols + 4;   // row pitch of hq
constexpr int kKtLd = kCols + 1;   // row pitch of kt

__host__ __device__ inline ConvLayout conv_layout(int r) {
  ConvLayout L;
  L.p_ld = 2 * r + 4;
  L.u = 0;                                   // [2][32][r] bf16 (bulk copy)
  L.vt = L.u + 2 * kCols * r * 2;            // [32][2r] bf16 (bulk copy; output sites with a next site)
  L.p = L.vt + kCols * 2 * r * 2;            // [16][p_ld] tf32
  L.x = L.p + kRows * L.p_ld * 4;            // [17][32] fp32: rows m0-1 .. m0+15
  L.hq = L.x + (kRows + 1) * kCols * 4;      // [16][36] tf32: x * g of the rows
  L.kt = L.hq + kRows * kHqLd * 4;           // [2][16][33] fp32: U_i P_t
  L.base = L.kt + 2 * kRows * kKtLd * 4;     // [2][32] fp32
  L.sc = L.base + 2 * kCols * 4;             // [17] row scales (32 slots)
  L.scp = L.sc + 32 * 4;                     // [17][8] partial sums of the scales
  L.total = L.scp + 17 * 8 * 4 + 16;
  return L;
}

__global__ void __launch_bounds__(kThreads) conv_apply_kernel(const __grid_constant__ ConvArgs a) {
  extern __shared__ __align__(16) uint8_t sm[];
  __shared__ __align__(8) uint64_t bar;
  const int r = a.r, r2 = 2 * r;
  const int h0 = blockIdx.x * kCols, m0 = blockIdx.y * kRows;
  const bool out_site = a.out_h == nullptr;
  const bool next = out_site && a.vt != nullptr;
  const ConvLayout L = conv_layout(r);
  const uint16_t* us = reinterpret_cast<const uint16_t*>(sm + L.u);
  const uint16_t* vts = reinterpret_cast<const uint16_t*>(sm + L.vt);
  uint32_t* ps = reinterpret_cast<uint32_t*>(sm + L.p);
  float* xs = reinterpret_cast<float*>(sm + L.x);
  uint32_t* hq = reinterpret_cast<uint32_t*>(sm + L.hq);
  float* kt = reinterpret_cast<float*>(sm + L.kt);
  float* bs = reinterpret_cast<float*>(sm + L.base);
  float* sc = reinterpret_cast<float*>(sm + L.sc);
  float* scp = reinterpret_cast<float*>(sm + L.scp);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, q = lane & 3;

  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {   // weight slices: U_0, U_1 rows h0..h0+31, and the next site's V^T rows
    const uint32_t ub = kCols * r * 2, vb = next ? kCols * r2 * 2 : 0;
    mbar_arrive_expect_tx(&bar, 2 * ub + vb);
    bulk_load(sm + L.u, a.U + static_cast<size_t>(h0) * r, ub, &bar);
    bulk_load(sm + L.u + kCols * r * 2, a.U + (static_cast<size_t>(a.H) + h0) * r, ub, &bar);
    if (next) bulk_load(sm + L.vt, a.vt + static_cast<size_t>(h0) * r2, vb, &bar);
  }
  if (tid < 2 * kCols) bs[tid] = bf16_to_f32(a.base[(tid / kCols) * a.H + h0 + (tid % kCols)]);
  grid_dep_wait();
  grid_dep_launch();

  // P rows and x rows m0-1 .. m0+15 (and, at input sites, the rows'
  // sums-of-squares parts), every load issued before the first use
  const int np = kRows * r2;
  float pv[8], xv[2];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int i = tid + k * kThreads, t = i / r2, j = i - t * r2, m = m0 + t;
    pv[k] = 0.f;
    if (i < np && m < a.M)
      pv[k] = out_site ? a.y[static_cast<size_t>(m) * a.ld_y + a.H + j] : a.P[static_cast<size_t>(m) * r2 + j];
  }
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int i = tid + k * kThreads, t = i / kCols, c = i % kCols, m = m0 - 1 + t;
    xv[k] = 0.f;
    if (i < (kRows + 1) * kCols && m >= 0 && m < a.M)
      xv[k] = out_site ? a.y[static_cast<size_t>(m) * a.ld_y + h0 + c]
                       : a.xin[static_cast<size_t>(m) * a.H + h0 + c] * bf16_to_f32(a.gin[h0 + c]);
  }
  if (!out_site) rms_scales(a.ss, a.ss_parts, a.ss_ld, m0 - 1, kRows + 1, a.M, a.inv_hidden, a.eps, scp, sc);
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int i = tid + k * kThreads, t = i / r2, j = i - t * r2;
    if (i < np) ps[t * L.p_ld + j] = to_tf32(out_site || a.p_scaled ? pv[k] : pv[k] * sc[t + 1]);
  }
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int i = tid + k * kThreads;
    if (i < (kRows + 1) * kCols) xs[i] = out_site ? xv[k] : xv[k] * sc[i / kCols];
  }
  // input sites: zero this CTA's share of the accumulator the next output site adds into
  if (!out_site && a.zero) {
    const int nb = gridDim.x * gridDim.y, b = blockIdx.y * gridDim.x + blockIdx.x;
    const size_t n = static_cast<size_t>(a.M) * r2, per = (n + nb - 1) / nb, z0 = b * per;
    for (size_t i = z0 + tid; i < min(n, z0 + per); i += kThreads) a.zero[i] = 0.f;
  }
  const bool ok = mbar_wait(&bar, 0);
  if (!ok) latch_status(a.status, kDevTimeout);
  if (!__syncthreads_and(ok)) return;

  // U_i P_t for the 16 rows x 32 columns: warp (tap, 8-column tile), r/8
  // tensor-core steps over the rank
  if (warp < 8) {
    const int tap = warp >> 2, nt = warp & 3;
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    const uint32_t* pa = ps + tap * r;
    const uint16_t* ub = us + (tap * kCols + nt * 8 + g) * r;
    for (int k0 = 0; k0 < r; k0 += 8) {
      const uint32_t af[4] = {pa[g * L.p_ld + k0 + q], pa[(g + 8) * L.p_ld + k0 + q], pa[g * L.p_ld + k0 + q + 4],
                              pa[(g + 8) * L.p_ld + k0 + q + 4]};
      mma_tf32(d, af, bf16_bits_f32(ub[k0 + q]), bf16_bits_f32(ub[k0 + q + 4]));
    }
    float* kd = kt + tap * kRows * kKtLd + nt * 8 + 2 * q;
    kd[g * kKtLd] = d[0];
    kd[g * kKtLd + 1] = d[1];
    kd[(g + 8) * kKtLd] = d[2];
    kd[(g + 8) * kKtLd + 1] = d[3];
  }
  __syncthreads();

  // the two taps for this thread's column and row; block position 0 of each
  // sequence has no predecessor
  const int col = tid & (kCols - 1), t = tid / kCols, m = m0 + t;
  const float xt = xs[(t + 1) * kCols + col];
  const float xp = (m % a.B) != 0 ? xs[t * kCols + col] : 0.f;
  const float o = (bs[col] + kt[t * kKtLd + col]) * xt + (bs[kCols + col] + kt[(kRows + t) * kKtLd + col]) * xp;
  const size_t off = static_cast<size_t>(m) * a.H + h0 + col;
  if (!out_site) {
    if (m < a.M) a.out_h[off] = f32_to_bf16(o);
    return;
  }
  float sq = 0.f, hv = 0.f;
  if (m < a.M) {
    const float xn = a.x[off] + o;
    const float gain = bf16_to_f32(a.gain[h0 + col]);
    a.x[off] = xn;
    a.out_hg[off] = f32_to_bf16(xn * gain);
    hv = xn * gain;
    sq = xn * xn;
  }
  hq[t * kHqLd + col] = to_tf32(hv);
  // the row's sum of x^2 over the 32 columns (one warp)
#pragma unroll
  for (int o2 = 16; o2 > 0; o2 >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o2);
  if (col == 0 && m < a.M) a.out_ss[static_cast<size_t>(blockIdx.x) * a.out_ss_ld + m] = sq;
  if (!next) return;
  __syncthreads();

  // the next input site's products over these columns, added into the
  // accumulator: acc[m][j] += sum_c (x * g)[m][c] V_next[j][c]; warp w takes
  // the 8-product tiles w, w + 16, ..., 4 tensor-core steps over the columns
  for (int nt = warp; nt < r2 / 8; nt += kThreads / 32) {
    float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k0 = 0; k0 < kCols; k0 += 8) {
      const uint32_t af[4] = {hq[g * kHqLd + k0 + q], hq[(g + 8) * kHqLd + k0 + q], hq[g * kHqLd + k0 + q + 4],
                              hq[(g + 8) * kHqLd + k0 + q + 4]};
      mma_tf32(d, af, bf16_bits_f32(vts[(k0 + q) * r2 + nt * 8 + g]), bf16_bits_f32(vts[(k0 + q + 4) * r2 + nt * 8 + g]));
    }
    const int j = nt * 8 + 2 * q;
    if (m0 + g < a.M) atomicAdd(reinterpret_cast<float2*>(a.pacc + static_cast<size_t>(m0 + g) * r2 + j), make_float2(d[0], d[1]));
    if (m0 + g + 8 < a.M)
      atomicAdd(reinterpret_cast<float2*>(a.pacc + static_cast<size_t>(m0 + g + 8) * r2 + j), make_float2(d[2], d[3]));
  }
}

// F[j][c] = sum_h V[j][h] W[h][c] (install time): 128 columns c and 32 rows j per CTA.
__global__ void __launch_bounds__(128) conv_fold_kernel(const uint16_t* V, const uint16_t* W, int J, int H, int K,
                                                         uint16_t* F) {
  __shared__ float vs[32][64];
  const int c = blockIdx.x * 128 + threadIdx.x, j0 = blockIdx.y * 32;
  float acc[32];
#pragma unroll
  for (int q = 0; q < 32; ++q) acc[q] = 0.f;
  for (int hb = 0; hb < H; hb += 64) {
    for (int i = threadIdx.x; i < 32 * 64; i += 128) {
      const int jj = i >> 6, hh = i & 63;
      vs[jj][hh] = j0 + jj < J && hb + hh < H ? bf16_to_f32(V[static_cast<size_t>(j0 + jj) * H + hb + hh]) : 0.f;
    }
    __syncthreads();
    if (c < K) {
      const int hn = min(64, H - hb);
      for (int hh = 0; hh < hn; ++hh) {
        const float w = bf16_to_f32(W[static_cast<size_t>(hb + hh) * K + c]);
#pragma unroll
        for (int q = 0; q < 32; ++q) acc[q] += vs[q][hh] * w;
      }
    }
    __syncthreads();
  }
  if (c < K) {
#pragma unroll
    for (int q = 0; q < 32; ++q)
      if (j0 + q < J) F[static_cast<size_t>(j0 + q) * K + c] = f32_to_bf16(acc[q]);
  }
}

// out[c][r] = in[r][c] for a rows x cols bf16 matrix (32 x 32 tiles).
__global__ void __launch_bounds__(256) transpose_bf16_kernel(const uint16_t* in, int rows, int cols, uint16_t* out) {
  __shared__ uint16_t t[32][33];
  const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
  for (int i = threadIdx.x; i < 32 * 32; i += 256) {
    const int rr = i >> 5, cc = i & 31;
    if (r0 + rr < rows && c0 + cc < cols) t[rr][cc] = in[static_cast<size_t>(r0 + rr) * cols + c0 + cc];
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 32 * 32; i += 256) {
    const int cc = i >> 5, rr = i & 31;
    if (r0 + rr < rows && c0 + cc < cols) out[static_cast<size_t>(c0 + cc) * rows + r0 + rr] = t[rr][cc];
  }
}

}  // namespace

size_t conv_smem_bytes(int r) { return static_cast<size_t>(conv_layout(r).total); }

cudaError_t launch_conv_apply(const ConvArgs& a, cudaStream_t s) {
  const int smem = conv_layout(a.r).total;
  if (smem > 48 * 1024) {
    static int configured = 0;
    if (!configured) {
      cudaError_t e = cudaFuncSetAttribute(conv_apply_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           conv_layout(kConvMaxRank).total);
      if (e != cudaSuccess) return e;
      configured = 1;
    }
  }
  const dim3 grid(a.H / kCols, (a.M + kRows - 1) / kRows);
  return launch_pdl(conv_apply_kernel, grid, dim3(kThreads), smem, s, a);
}

cudaError_t launch_conv_fold(const uint16_t* V, const uint16_t* W, int J, int H, int K, uint16_t* F, cudaStream_t s) {
  const dim3 grid((K + 127) / 128, (J + 31) / 32);
  conv_fold_kernel<<<grid, 128, 0, s>>>(V, W, J, H, K, F);
  return cudaGetLastError();
}

cudaError_t launch_transpose_bf16(const uint16_t* in, int rows, int cols, uint16_t* out, cudaStream_t s) {
  const dim3 grid((cols + 31) / 32, (rows + 31) / 32);
  transpose_bf16_kernel<<<grid, 256, 0, s>>>(in, rows, cols, out);
  return cudaGetLastError();
}

}  // namespace dfl
