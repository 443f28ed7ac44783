// sampling.cu - temperature sampling with top-k / top-p filters and the
// lossless speculative-sampling verify ("DFlash - Block Diffusion for Flash
// Speculative Decoding" notes, 6.2 "Sampling (Temperature = 1)" and the
// "Lossless Guarantee"; the "DFlash 2" notes evaluate at temperature 1,
// top-p 0.95, top-k 20 with lossless rejection sampling).
//
// A filtered distribution keeps the top_k largest logits (topk.cuh gives the
// 32 largest of each row; ties to the lower id), takes their temperature
// softmax, keeps the shortest prefix whose mass reaches top_p and
// renormalises. Lists are 32 wide: ids in decreasing probability, -1 and 0
// past the kept entries.
//
//   sample_filter_kernel   one CTA per row: merge the row's slice lists,
//                          filter, and (with uniforms) draw by inverse CDF;
//   verify_sample_kernel   one warp per sequence: walking the block, accept
//                          draft x_j when u_j < min(1, p_j(x_j) / q_j(x_j)),
//                          else draw from max(0, p_j - q_j); after B - 1
//                          acceptances draw the bonus from p_{B-1}; then
//                          commit min(tau, pending) pending tokens.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"
#include "topk.cuh"

namespace dfl {
namespace {

constexpr int kW = kSampleWidth;   // list width (32)
constexpr int kFilterThreads = 256;

__device__ __forceinline__ float warp_incl_scan(float v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  return v;
}

// First lane whose inclusive cumulative weight exceeds u * total among lanes
// with `real`; the last real lane when rounding leaves none (as the oracle's
// draw clamps to the list's end).
__device__ __forceinline__ int draw_lane(float c, float total, float u, bool real) {
  const uint32_t m = __ballot_sync(0xffffffffu, real && c > u * total);
  if (m) return __ffs(m) - 1;
  const uint32_t rl = __ballot_sync(0xffffffffu, real);
  return rl ? 31 - __clz(rl) : 0;
}

__global__ void __launch_bounds__(kFilterThreads) sample_filter_kernel(const __grid_constant__ FilterArgs a) {
  __shared__ unsigned long long s_keys[kSampleMaxSlices * kW], s_kept[kSampleMaxSlices * kW];
  __shared__ unsigned long long s_top[kW];
  __shared__ unsigned long long s_thr, s_lo;
  __shared__ int s_m;
  grid_dep_wait();
  grid_dep_launch();
  const int r = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
  topk::merge_lists<kW>(a.part + static_cast<size_t>(r) * a.slices * kW, a.slices, tid, kFilterThreads, s_keys,
                        s_kept, &s_thr, &s_lo, &s_m, s_top, [] { __syncthreads(); });
  if (tid >= 32) return;
  const unsigned long long k = s_top[lane];
  const bool valid = k != 0 && lane < a.top_k;
  const float l = topk::key_value(k);
  const int id = topk::key_col(k);
  const float l0 = __shfl_sync(0xffffffffu, l, 0);
  const float w = valid ? expf((l - l0) * a.inv_temperature) : 0.f;
  const float c = warp_incl_scan(w, lane);
  const float total = __shfl_sync(0xffffffffu, c, 31);
  // keep while the mass before the entry is below top_p (the entry that
  // reaches top_p is kept)
  const bool keep = valid && (lane == 0 || c - w < a.top_p * total);
  const float w2 = keep ? w : 0.f;
  const float c2 = warp_incl_scan(w2, lane);
  const float total2 = __shfl_sync(0xffffffffu, c2, 31);
  const size_t o = static_cast<size_t>(r) * kW + lane;
  a.out_ids[o] = keep ? id : -1;
  a.out_probs[o] = keep ? w2 / total2 : 0.f;
  if (a.drawn) {
    const int pick = draw_lane(c2, total2, a.uniforms[r], keep);
    const int did = __shfl_sync(0xffffffffu, id, pick);
    if (lane == 0) a.drawn[r] = did;
  }
}

// p(x) for the id x in a 32-wide list held one entry per lane.
__device__ __forceinline__ float prob_in(int my_id, float my_p, int x) {
  const uint32_t m = __ballot_sync(0xffffffffu, my_id >= 0 && my_id == x);
  const float v = __shfl_sync(0xffffffffu, my_p, m ? __ffs(m) - 1 : 0);
  return m ? v : 0.f;
}

__global__ void verify_sample_kernel(const __grid_constant__ SeqMeta meta, SeqState st,
                                     const __grid_constant__ VerifySampleArgs a) {
  grid_dep_wait();
  grid_dep_launch();
  const int i = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (i >= meta.n_seq) return;
  const int B = meta.B, T = B - 1;
  int acc = T, tok = -1;
  for (int j = 0; j < T; ++j) {
    const int x = a.drafts[static_cast<size_t>(i) * T + j];
    const size_t pq = (static_cast<size_t>(i) * B + j) * kW + lane;
    const size_t qq = (static_cast<size_t>(i) * T + j) * kW + lane;
    const int pid = a.p_ids[pq], qid = a.q_ids[qq];
    const float pp = a.p_probs[pq], qp = a.q_probs[qq];
    const float px = prob_in(pid, pp, x), qx = prob_in(qid, qp, x);
    const float ua = a.u_accept[static_cast<size_t>(i) * T + j];
    if (qx > 0.f && ua < fminf(1.f, px / qx)) continue;
    // rejected: draw from max(0, p - q) in p's order
    float qv = 0.f;
#pragma unroll 8
    for (int s = 0; s < 32; ++s) {
      const int sid = __shfl_sync(0xffffffffu, qid, s);
      const float sp = __shfl_sync(0xffffffffu, qp, s);
      if (pid >= 0 && sid == pid) qv = sp;
    }
    const float rr = pid >= 0 ? fmaxf(0.f, pp - qv) : 0.f;
    const float c = warp_incl_scan(rr, lane);
    const float total = __shfl_sync(0xffffffffu, c, 31);
    const int pick = draw_lane(c, total, a.u_resample[static_cast<size_t>(i) * B + j], pid >= 0);
    tok = __shfl_sync(0xffffffffu, pid, pick);
    acc = j;
    break;
  }
  if (tok < 0) {   // every draft accepted: the bonus from p_{B-1}
    const size_t pq = (static_cast<size_t>(i) * B + T) * kW + lane;
    const int pid = a.p_ids[pq];
    const float pp = pid >= 0 ? a.p_probs[pq] : 0.f;
    const float c = warp_incl_scan(pp, lane);
    const float total = __shfl_sync(0xffffffffu, c, 31);
    const int pick = draw_lane(c, total, a.u_resample[static_cast<size_t>(i) * B + T], pid >= 0);
    tok = __shfl_sync(0xffffffffu, pid, pick);
    acc = T;
  }
  if (lane == 0) {
    a.tau[i] = acc + 1;
    a.bonus[i] = tok;
    if (tok < 0) latch_status(a.status, kDevBounds);   // an empty target list
    const int slot = meta.slot[i];
    const int p = st.pend[slot];
    st.len[slot] += min(acc + 1, p);
    st.pend[slot] = 0;
  }
}

}  // namespace

cudaError_t launch_sample_filter(const void* logits, bool bf16, int ld, int V, int rows, int draft_B,
                                 unsigned long long* part, const FilterArgs& fa, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  cudaError_t e;
  if (bf16) {
    e = launch_pdl(topk::topk_slices_kernel<uint16_t, kW, false>, dim3(fa.slices, rows), dim3(topk::kThreads), 0, s,
                   static_cast<const uint16_t*>(logits), ld, V, 0, part);
  } else {
    e = launch_pdl(topk::topk_slices_kernel<float, kW, true>, dim3(fa.slices, rows), dim3(topk::kThreads), 0, s,
                   static_cast<const float*>(logits), ld, V, draft_B, part);
  }
  if (e != cudaSuccess) return e;
  return launch_pdl(sample_filter_kernel, dim3(rows), dim3(kFilterThreads), 0, s, fa);
}

int sample_slice_cols(bool bf16) { return bf16 ? topk::In<uint16_t>::kSliceCols : topk::In<float>::kSliceCols; }

cudaError_t launch_verify_sample(const SeqMeta& meta, SeqState st, const VerifySampleArgs& a, cudaStream_t s) {
  const int warps = 4;
  return launch_pdl(verify_sample_kernel, dim3((meta.n_seq + warps - 1) / warps), dim3(warps * 32), 0, s, meta, st, a);
}

}  // namespace dfl
