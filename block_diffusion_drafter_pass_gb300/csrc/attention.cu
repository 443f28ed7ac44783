// attention.cu - block attention over the injected context (non-causal, the
// drafter) or over the target's own cache (causal within the block).
//
// For each sequence and kv head, the G*B query rows of the block (G query
// heads per kv head, B block positions) attend to every committed context key
// of that layer (paged, 64 tokens per page) and to the block's own B keys:
// all of them in the drafter's non-causal pass; keys 0..j of the block for
// block position j in the target's causal pass (AttnArgs::causal).
//
// The keys are split into chunks of whole 64-key tiles (flash-decoding). A
// persistent grid, one CTA per SM, runs the (sequence, kv head, chunk) work
// items the host dealt to each CTA (largest first, to the least loaded CTA).
// Per CTA:
//   warp 0     TMA producer: the item's queries once, then per step of two
//              64-key units the key rows [64][d] and the transposed value
//              rows [d][64] of two pages (values are stored transposed in the
//              pool so that both products read K-major, 128-byte-swizzled
//              operands);
//   warp 1     allocates tensor memory and issues tcgen05.mma from one
//              thread: S = Q K^T (M = 128 query rows, N = 128 keys) into one
//              of two TMEM S buffers, then O += P V (N = d) into the item's
//              TMEM O buffer; Q and P are the A operand read from TMEM, so
//              shared memory feeds only K and V;
//   warp 6     L2 prefetch of the context pages a few steps ahead of warp 0;
//   warps 2-5  the softmax: online softmax in the log2 domain on S read from
//              TMEM, P written over its own S as packed bf16, O rescaled in
//              TMEM only when the row maximum grows by more than 2^8 (the
//              stale maximum is a valid reference point: P and O stay
//              bounded by 256x).
// S_{t+1} is issued before P_t is ready, so the softmax of one tile overlaps
// the products of the next. Each item leaves an unnormalised partial (O,
// running max, running sum); attn_combine_kernel merges the chunks of a row.
// Query row r of an item is (block position j, head g of the group) with
// r = j*G + g (the order the 3D query box lands in shared memory).
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace dfl {
namespace {

constexpr int kKeyTile = 64;
constexpr float kRescaleLog2 = 8.f;   // rescale O when the row max grows by more than 2^8
constexpr int kThreads = 224;         // producer, MMA, 4 softmax warps, L2 prefetch warp
constexpr int kConvWarps = 8;         // 8-bit pages: warps 8..15 (two warpgroups) convert the codes
                                      // to fp16 tiles; warp 7 idles
template <bool Q8>
constexpr int attn_threads() { return Q8 ? 256 + 32 * kConvWarps : kThreads; }
// 8-bit pages: the block is launched at 128 registers a thread (512 threads,
// the whole register file); warpgroups 0-1 (producer, MMA, softmax, loader)
// raise theirs to 168 and warpgroups 2-3 (converters) drop to 88, which sum
// to the launch's 65536.
constexpr uint32_t kQ8RegsMain = 168, kQ8RegsConv = 88;
static_assert(256 * kQ8RegsMain + 256 * kQ8RegsConv == 512 * 128, "register split of the 8-bit kernel");
constexpr int kPrefetchSteps = 4;     // the prefetch warp runs this many steps ahead of the producer

// Rows of the block's own key box: B rounded up to 16 or 32.
__host__ __device__ __forceinline__ int block_rows(int B) { return B <= 16 ? 16 : 32; }

template <int D, bool Q8 = false>
struct ACfg {
  // One pipeline stage holds one step: two 64-key units (context pages or the
  // block) as [K dim-box 0: 128 keys x 128 B]...[K dim-box D/64-1][V^T unit 0]
  // [V^T unit 1], so S = Q K^T of a step is one N = 128 product per K slice.
  // 8-bit pages: the raw loader brings each context unit as a raw region
  // (codes and scales, q8_head_bytes) into one of kRawSlots unit slots, as
  // far ahead as free slots allow, and the converter warps write the fp16
  // stage from them.
  static constexpr int kStages = Q8 ? (D == 128 ? 2 : 4) : (D == 128 ? 3 : 6);
  static constexpr int kUnitBox = 64 * 128;               // 64 rows x 128 bytes
  static constexpr int kKBox = 2 * kUnitBox;              // 128 key rows of one 64-dim slice
  static constexpr int kKBytes = (D / 64) * kKBox;
  static constexpr int kVUnit = (D / 64) * kUnitBox;      // values transposed [D][64] of one unit
  static constexpr int kStageBytes = kKBytes + 2 * kVUnit;
  static constexpr int kRawUnit = static_cast<int>(q8_head_bytes(D));
  // as many unit slots as the shared memory left by the stages holds (4 KB
  // under the 227 KB a block may use, kept for the static shared variables)
  static constexpr int kRawSlots = Q8 ? (227 * 1024 - 4096 - 1024 - kStages * kStageBytes) / kRawUnit : 0;
  static constexpr int kSmem = kStages * kStageBytes + kRawSlots * kRawUnit + 1024;
  static_assert(!Q8 || kRawSlots >= 4, "8-bit pages need at least two steps of raw slots");
  // TMEM columns: S buffers at 0 and 128 (P overwrites the first 64 columns
  // of its own S as packed bf16), Q at 256 (D/2 columns of packed bf16), O after it.
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kSCols = 2 * kKeyTile;
  static constexpr uint32_t kQCol = 2 * kSCols;
  static constexpr uint32_t kOCol = kQCol + D / 2;
  // 8-bit pages run the products in fp16 (Q, P and the decoded K/V tiles),
  // so that a code pair decodes in three packed instructions
  static constexpr uint32_t kIdescS = Q8 ? idesc_f16_f32(128, 2 * kKeyTile) : idesc_bf16_f32(128, 2 * kKeyTile);
  static constexpr uint32_t kIdescO = Q8 ? idesc_f16_f32(128, D) : idesc_bf16_f32(128, D);
};

// D[tmem] (+)= A[tmem] * B[smem]^T: A (M rows in TMEM lanes, K packed two bf16
// per 32-bit column), B from a shared-memory descriptor. One thread issues.
__device__ __forceinline__ void tc_mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

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

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
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
__device__ __forceinline__ void tmem_ld_half64(uint32_t taddr, float (&v)[64]) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.16x32bx2.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
      "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64], %65;\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
        "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
        "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr), "n"(SPLIT)
      : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
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

// 32x32b stores of packed words (one lane per thread), x16 / x32 columns.
__device__ __forceinline__ void tmem_st_u16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st_u32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
// 16x32bx2 stores of packed words: threads 0-15 to columns [c, c+n), threads
// 16-31 to [c+SPLIT, c+SPLIT+n) of the same 16 lanes.
template <int SPLIT>
__device__ __forceinline__ void tmem_st_half_u16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x32bx2.x16.b32 [%0], %17, {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "n"(SPLIT)
      : "memory");
}
template <int SPLIT>
__device__ __forceinline__ void tmem_st_half_u32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x32bx2.x32.b32 [%0], %33, {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31]), "n"(SPLIT)
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

// 8-bit pages: two codes of a stored offset-binary word (code + 128 per byte),
// selected by `sel`, decoded in fp16 and scaled by the fp16 pair s2. The
// byte under an fp16 exponent of 2^10 reads as 1024 + code + 128 exactly; one
// exact subtraction gives the code, one multiply applies the scale (rounded
// to fp16).
__device__ __forceinline__ uint32_t q8_pair_f16(uint32_t ub, uint32_t sel, uint32_t s2) {
  const uint32_t h = __byte_perm(ub, 0x64646464u, sel);
  const __half2 q = __hsub2(*reinterpret_cast<const __half2*>(&h), __halves2half2(__ushort_as_half(0x6480),
                                                                                  __ushort_as_half(0x6480)));
  const __half2 r = __hmul2(q, *reinterpret_cast<const __half2*>(&s2));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// 16 codes (one 16-byte word) with their fp16 scales (one pair per code pair)
// -> 8 fp16 pairs.
__device__ __forceinline__ void q8_decode16(const uint4& cw, const uint32_t (&s2)[8], uint32_t (&o)[8]) {
  const uint32_t w[4] = {cw.x, cw.y, cw.z, cw.w};   // stored offset-binary
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    o[2 * k] = q8_pair_f16(w[k], 0x4140u, s2[2 * k]);
    o[2 * k + 1] = q8_pair_f16(w[k], 0x4342u, s2[2 * k + 1]);
  }
}

// Shared-memory accesses by 32-bit shared-window address (the stage and raw
// ring pointers are realigned through an integer, which hides their state
// space from the compiler; generic accesses would cost 64-bit address math
// and the long scoreboard).
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds16(uint32_t a) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ void sts128(uint32_t a, const uint4& v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w));
}

// One 64-key context unit: raw region (K codes [64][D], V codes [D][64], K
// scales [64][D/32], V scales [D/32][64]) -> unit u of an fp16 stage in the
// 128-byte-swizzled layout the MMAs read (keys: row u*64 + k of each 64-dim
// slice box; transposed values: row r of box r/64 of the unit's V^T tile).
// Thread ct of NCT takes tasks ct + j*NCT, all in one unrolled round: the
// loads of every task first, then decode and stores (a converter warp is
// latency-bound, so its tasks must be independent in flight). raw and stage
// are shared-window addresses.
// Key task -> (key k, 16-dim group g). The eight tasks of one 16-byte access
// phase of a warp take two keys, the first key's four groups of one 64-dim
// box and the second key's four of the other box (d = 64: one box, the two
// keys 64 bytes apart): their code loads cover the two halves of the banks,
// and their swizzled stores land in distinct chunks (even and odd rows).
template <int D>
__device__ __forceinline__ void q8_key_task(int task, int& k, int& g) {
  if constexpr (D == 128) {
    const int kp = task >> 4, b = (task >> 3) & 1, w = task & 7, par = w >> 2;
    k = 2 * kp + par;
    g = ((b ^ par) << 2) + (w & 3);
  } else {
    static_assert(D == 64, "head dims 64 and 128");
    const int kp = task >> 3, w = task & 7;
    k = 2 * kp + (w >> 2);
    g = w & 3;
  }
}

template <int D, int NCT, int kKBox, int kKBytes, int kVUnit, int kUnitBox>
__device__ __forceinline__ void q8_convert_unit(uint32_t raw, uint32_t stage, int u, int ct) {
  // keys: tasks (key k, 16-dim group g); values: tasks (dim r, 16-key group kg)
  constexpr int kTK = 64 * (D / 16), kTV = D * 4, kIlp = (kTK + kTV) / NCT;
  static_assert(kTK % NCT == 0 && kTV % NCT == 0, "each round takes only keys or only values");
  const uint32_t ksc = raw + static_cast<uint32_t>(q8_kscale_off(D));
  const uint32_t vsc = raw + static_cast<uint32_t>(q8_vscale_off(D));
  const uint32_t vcd = raw + static_cast<uint32_t>(q8_vcode_off(D));
  uint4 cw[kIlp];
  uint32_t s2[kIlp][8];
#pragma unroll
  for (int j = 0; j < kIlp; ++j) {
    const int task = ct + j * NCT;
    if (j * NCT < kTK) {
      int k, g;
      q8_key_task<D>(task, k, g);
      cw[j] = lds128(raw + k * D + g * 16);
      const uint32_t s1 = lds16(ksc + (k * (D / 32) + (g >> 1)) * 2);
#pragma unroll
      for (int c = 0; c < 8; ++c) s2[j][c] = s1 | (s1 << 16);
    } else {
      const int r = (task - kTK) >> 2, kg = (task - kTK) & 3;
      cw[j] = lds128(vcd + r * 64 + kg * 16);
      // the 16 keys' scales of this dim's block: 8 fp16 pairs, 32 contiguous bytes
      const uint32_t sp = vsc + ((r >> 5) * 64 + kg * 16) * 2;
      const uint4 sa = lds128(sp), sb = lds128(sp + 16);
      s2[j][0] = sa.x; s2[j][1] = sa.y; s2[j][2] = sa.z; s2[j][3] = sa.w;
      s2[j][4] = sb.x; s2[j][5] = sb.y; s2[j][6] = sb.z; s2[j][7] = sb.w;
    }
  }
#pragma unroll
  for (int j = 0; j < kIlp; ++j) {
    const int task = ct + j * NCT;
    uint32_t o[8];
    q8_decode16(cw[j], s2[j], o);
    const uint4 lo = make_uint4(o[0], o[1], o[2], o[3]), hi = make_uint4(o[4], o[5], o[6], o[7]);
    if (j * NCT < kTK) {
      int k, g;
      q8_key_task<D>(task, k, g);
      const int row = u * 64 + k, c0 = (g & 3) * 2;
      const uint32_t rowp = stage + (g >> 2) * kKBox + row * 128;
      sts128(rowp + ((c0 ^ (row & 7)) << 4), lo);
      sts128(rowp + (((c0 + 1) ^ (row & 7)) << 4), hi);
    } else {
      const int r = (task - kTK) >> 2, kg = (task - kTK) & 3;
      const int row = r & 63, c0 = kg * 2;
      const uint32_t rowp = stage + kKBytes + u * kVUnit + (r >> 6) * kUnitBox + row * 128;
      sts128(rowp + ((c0 ^ (row & 7)) << 4), lo);
      sts128(rowp + (((c0 + 1) ^ (row & 7)) << 4), hi);
    }
  }
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
  int i, kvh, tb, te;   // sequence index, kv head, units [tb, te)
  int slot;             // partial-buffer slot: (sequence, kv head, chunk) in row-major order
};

// SPREAD (G*B <= 64): query row r sits in TMEM lane 32*(r/16) + r%16, so all
// four lane quarters (and the four SM sub-partitions that own them) carry 16
// rows, and two threads share a row (64 keys of a step each). Otherwise one
// thread per row, row r in lane r.
//
// Units are 64-key tiles: context pages 0 .. n_ctx-1, then the block (unit
// n_ctx). An item covers units [tb, te) with tb even; a step takes units
// (tb + 2j, tb + 2j + 1), the second possibly absent.
template <int D, bool SPREAD, bool Q8>
__global__ void __launch_bounds__(attn_threads<Q8>(), 1)
    attn_kernel(const __grid_constant__ AttnMaps maps, const __grid_constant__ AttnArgs a,
                const __grid_constant__ AttnSched sched) {
  using C = ACfg<D, Q8>;
  constexpr int S = C::kStages;
  constexpr int RS = Q8 ? C::kRawSlots : 1;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* raw_ring = smem + S * C::kStageBytes;   // 8-bit pages: kRawSlots raw unit slots
  __shared__ __align__(8) uint64_t kv_full[S], kv_empty[S];
  __shared__ __align__(8) uint64_t raw_full[RS], raw_empty[RS];
  __shared__ __align__(8) uint64_t q_ready, mma_done, o_full, o_free;
  __shared__ __align__(8) uint64_t s_full[2], p_full[2];
  __shared__ uint32_t tmem_slot;
  __shared__ int s_prefix[kMaxBatch + 1];
  __shared__ int s_len[kMaxBatch];
  __shared__ int s_nctx[kMaxBatch];
  __shared__ int s_nch[kMaxBatch];
  __shared__ volatile int abort_flag;
  __shared__ volatile int s_issued;   // steps whose copies the producer has issued

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_seq = a.meta.n_seq, B = a.meta.B;
  const int nkv = a.n_kv_heads, G = a.n_q_heads / a.n_kv_heads;
  const int R = G * B;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&kv_full[s], Q8 ? 1 + kConvWarps : 1);   // producer (+ converter warps)
      mbar_init(&kv_empty[s], 1);
    }
    for (int r = 0; r < RS; ++r) {
      mbar_init(&raw_full[r], 1);
      mbar_init(&raw_empty[r], kConvWarps);
    }
    mbar_init(&q_ready, 4);
    mbar_init(&mma_done, 1);
    mbar_init(&o_full, 1);
    s_issued = 0;
    mbar_init(&o_free, 4);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&p_full[b], 4);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&maps.pool_k);
    tma_prefetch_desc(&maps.pool_vt);
    tma_prefetch_desc(&maps.kblk);
    tma_prefetch_desc(&maps.vblk);
  }
  if (warp == 1) tmem_alloc(&tmem_slot, C::kTmemCols);
  // Dependencies: every launch sequence of the library puts a kernel that
  // waits for its predecessor before it lets its dependents start (the block
  // embedding, the previous layer's combine) between the last writer of the
  // KV pool, page table and lengths and this kernel. They are final when this
  // kernel starts, so the context pages stream before griddepcontrol.wait;
  // only q and the block's own keys and values, written by the projection
  // kernel just before, are read after it (producer: block unit; softmax
  // warps: q).
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

  // This CTA's records: every role walks the same list and skips the same
  // records (chunks the device's lengths do not reach).
  const int rec_end = sched.off[blockIdx.x + 1];
  auto rec_ok = [&](int k) {
    const uint32_t w = sched.item[k];
    const int i = static_cast<int>(w >> 24), h = static_cast<int>((w >> 16) & 0xFFu);
    return i < n_seq && h < nkv && static_cast<int>(w & 0xFFFFu) < s_nch[i];
  };
  auto next_rec = [&](int k) {
    while (k < rec_end && !rec_ok(k)) ++k;
    return k;
  };
  const int rec_begin = next_rec(sched.off[blockIdx.x]);
  auto decode = [&](int k) {
    const uint32_t w = sched.item[k];
    Item it;
    it.i = static_cast<int>(w >> 24);
    it.kvh = static_cast<int>((w >> 16) & 0xFFu);
    const int chunk = static_cast<int>(w & 0xFFFFu);
    it.tb = chunk * a.chunk_tiles;
    it.te = min(s_nctx[it.i] + 1, it.tb + a.chunk_tiles);
    it.slot = s_prefix[it.i] + it.kvh * s_nch[it.i] + chunk;
    return it;
  };
  auto give_up = [&]() {
    abort_flag = 1;
    latch_status(a.status, kDevTimeout);
  };

  // The converter warpgroups and the rest each change their register count
  // once, at the top of their branch (every warp of a warpgroup executes the
  // same instruction), so each role is compiled against its own budget.
  if (Q8 && warp >= 8) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kQ8RegsConv) : "memory");
    // ---------------- 8-bit page converters ----------------
    // Walk the producer's steps: wait for a free stage; per context unit of
    // the step, wait for its raw slot (context units are numbered in walk
    // order, as the raw loader issues them), decode it into the stage and free
    // the slot; then make the stores visible to the tensor cores and arrive on
    // the stage (the producer's arrival counts the block unit's copies).
    const int ct = threadIdx.x - 8 * 32;
    int q = 0, qu = 0;
    bool dead = false;
    for (int rk = rec_begin; rk < rec_end && !dead; rk = next_rec(rk + 1)) {
      const Item it = decode(rk);
      const int nctx = s_nctx[it.i];
      for (int t0 = it.tb; t0 < it.te && !dead; t0 += 2, ++q) {
        const int s = q % S;
        if (!__all_sync(0xffffffffu, mbar_wait(&kv_empty[s], ((q / S) & 1) ^ 1, &abort_flag))) {
          give_up();
          dead = true;
          break;
        }
        const int nu = min(2, it.te - t0);
        for (int u = 0; u < nu; ++u) {
          if (t0 + u >= nctx) continue;
          const int r = qu % RS;
          if (!__all_sync(0xffffffffu, mbar_wait(&raw_full[r], (qu / RS) & 1, &abort_flag))) {
            give_up();
            dead = true;
            break;
          }
          q8_convert_unit<D, 32 * kConvWarps, C::kKBox, C::kKBytes, C::kVUnit, C::kUnitBox>(
              smem_u32(raw_ring + r * C::kRawUnit), smem_u32(smem + s * C::kStageBytes), u, ct);
          __syncwarp();
          if (lane == 0) mbar_arrive(&raw_empty[r]);
          ++qu;
        }
        if (dead) break;
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&kv_full[s]);
      }
    }
  } else {
    if constexpr (Q8) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kQ8RegsMain) : "memory");
  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      const int Bb = block_rows(B);
      int q = 0;
      bool dead = false, waited = false;
      for (int rk = rec_begin; rk < rec_end && !dead; rk = next_rec(rk + 1)) {
        const Item it = decode(rk);
        const int slot = a.meta.slot[it.i], nctx = s_nctx[it.i];
        const int* ptab = a.seqs.page_table + static_cast<size_t>(slot) * a.seqs.pages_per_seq;
        auto page_of = [&](int t) {   // -1 (latched below) if the table is too short
          return t < nctx ? (t < a.seqs.pages_per_seq ? ptab[t] : -1) : 0;
        };
        int cur0 = page_of(it.tb), cur1 = it.tb + 1 < it.te ? page_of(it.tb + 1) : 0;
        for (int t0 = it.tb; t0 < it.te; t0 += 2, ++q) {
          // page ids of the next step are in flight during the wait below
          const int nxt0 = t0 + 2 < it.te ? page_of(t0 + 2) : 0;
          const int nxt1 = t0 + 3 < it.te ? page_of(t0 + 3) : 0;
          const int s = q % S;
          if (!mbar_wait(&kv_empty[s], ((q / S) & 1) ^ 1, &abort_flag)) {
            give_up();
            dead = true;
            break;
          }
          uint8_t* st = smem + s * C::kStageBytes;
          const int nu = min(2, it.te - t0);
          uint32_t bytes = 0;
          for (int u = 0; u < nu; ++u) {
            if (t0 + u < nctx) bytes += Q8 ? 0 : 2 * C::kVUnit;
            else bytes += (D / 64) * Bb * 128 + C::kVUnit;
          }
          mbar_arrive_expect_tx(&kv_full[s], bytes);
          for (int u = 0; u < nu; ++u) {
            const int t = t0 + u;
            uint8_t* ku = st + u * C::kUnitBox;
            uint8_t* vu = st + C::kKBytes + u * C::kVUnit;
            if (t < nctx) {
              if constexpr (Q8) continue;   // written by the converter warps
              int page = u == 0 ? cur0 : cur1;
              if (page < 0 || page >= a.pool_pages) {
                latch_status(a.status, kDevBounds);
                page = 0;
              }
              const int lp = a.layer * a.pool_pages + page;
              const int rowk = (lp * 2 * nkv + it.kvh) * kKeyTile;   // rows of d elements
              const int rowv = ((lp * 2 + 1) * nkv + it.kvh) * D;    // rows of 64 elements
#pragma unroll
              for (int bx = 0; bx < D / 64; ++bx) {
                tma_load_2d(ku + bx * C::kKBox, &maps.pool_k, &kv_full[s], bx * 64, rowk);
                tma_load_2d(vu + bx * C::kUnitBox, &maps.pool_vt, &kv_full[s], 0, rowv + bx * 64);
              }
            } else {
              if (!waited) {   // the block's keys and values come from the projection kernel
                grid_dep_wait();
                waited = true;
              }
#pragma unroll
              for (int bx = 0; bx < D / 64; ++bx) {
                tma_load_3d(ku + bx * C::kKBox, &maps.kblk, &kv_full[s], bx * 64, it.kvh, it.i * B);
                tma_load_2d(vu + bx * C::kUnitBox, &maps.vblk, &kv_full[s], 0,
                            (it.i * nkv + it.kvh) * D + bx * 64);
              }
            }
          }
          s_issued = q + 1;
          cur0 = nxt0;
          cur1 = nxt1;
        }
      }
      // copies still in flight complete before shared memory is released
      for (int j = max(0, q - S); j < q; ++j) mbar_wait(&kv_full[j % S], (j / S) & 1);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    // Per step q: S_{q+1} is issued before PV_q, so S of the next step
    // overlaps the softmax of this one. P_q lives in S buffer q&1; S_{q+2}
    // overwrites it only after PV_q, which precedes it in issue order.
    if (lane == 0) {
      const uint32_t kv_base = smem_u32(smem);
      auto issue_s = [&](int q) {   // S[q & 1] = Q K^T over the step's 128 keys
        const uint32_t kb = kv_base + (q % S) * C::kStageBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          tc_mma_bf16_ts(tmem + (q & 1) * C::kSCols, tmem + C::kQCol + kk * 8,
                         sdesc_kmajor_sw128(kb + (kk >> 2) * C::kKBox + (kk & 3) * 32), C::kIdescS, kk > 0);
        tc_commit(&s_full[q & 1]);
      };
      auto issue_pv = [&](int q, int j, const Item& it) {   // O += P V over the step's units
        const int nu = min(2, it.te - (it.tb + 2 * j));
        const uint32_t vb = kv_base + (q % S) * C::kStageBytes + C::kKBytes;
        for (int u = 0; u < nu; ++u) {
#pragma unroll
          for (int kk = 0; kk < kKeyTile / 16; ++kk)
            tc_mma_bf16_ts(tmem + C::kOCol, tmem + (q & 1) * C::kSCols + u * 32 + kk * 8,
                           sdesc_kmajor_sw128(vb + u * C::kVUnit + kk * 32), C::kIdescO,
                           (j > 0 || u > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(&kv_empty[q % S]);
      };
      int q = 0, k = 0;
      bool dead = false;
      for (int rk = rec_begin; rk < rec_end && !dead; rk = next_rec(rk + 1), ++k) {
        const Item it = decode(rk);
        const int ns = (it.te - it.tb + 1) >> 1;
        if (!mbar_wait(&q_ready, k & 1, &abort_flag)) {
          give_up();
          break;
        }
        // Issue whichever product is ready, PV first (it frees a stage):
        // S_x needs its keys and PV_{x-2} issued (P_{x-2} lives in S buffer
        // x&1); PV_y needs P_y (and, first in the item, O read out).
        int ns_done = 0, npv = 0;
        unsigned long long t0 = global_ns();
        while (npv < ns) {
          bool moved = false;
          if (npv < ns_done && mbar_test_wait(&p_full[(q + npv) & 1], ((q + npv) >> 1) & 1) &&
              (npv > 0 || mbar_test_wait(&o_free, (k & 1) ^ 1))) {
            tc_fence_after();
            issue_pv(q + npv, npv, it);
            ++npv;
            moved = true;
          }
          if (ns_done < ns && ns_done <= npv + 1 &&
              mbar_test_wait(&kv_full[(q + ns_done) % S], ((q + ns_done) / S) & 1)) {
            tc_fence_after();
            issue_s(q + ns_done);
            ++ns_done;
            moved = true;
          }
          if (moved) {
            t0 = global_ns();
          } else if (abort_flag || global_ns() - t0 > kWaitLimitNs) {
            give_up();
            dead = true;
            break;
          }
        }
        if (dead) break;
        tc_commit(&o_full);
        q += ns;
      }
      // every issued MMA completes before TMEM and shared memory are released
      tc_commit(&mma_done);
      mbar_wait(&mma_done, 0);
    }
  } else if (Q8 && warp == 7) {   // idle: the converters take whole warpgroups
  } else if (Q8 && warp == 6) {
    // ---------------- 8-bit page raw loader ----------------
    // Walks the same context units in the same order and brings each raw
    // region (codes and scales of one page and kv head) into the next unit
    // slot with one bulk copy, as soon as the converters have freed it.
    if (lane == 0) {
      int qu = 0;
      bool dead = false;
      for (int rk = rec_begin; rk < rec_end && !dead; rk = next_rec(rk + 1)) {
        const Item it = decode(rk);
        const int slot = a.meta.slot[it.i], nctx = s_nctx[it.i];
        const int* ptab = a.seqs.page_table + static_cast<size_t>(slot) * a.seqs.pages_per_seq;
        const int t_end = min(it.te, nctx);
        for (int t = it.tb; t < t_end; ++t, ++qu) {
          const int r = qu % RS;
          if (!mbar_wait(&raw_empty[r], ((qu / RS) & 1) ^ 1, &abort_flag)) {
            give_up();
            dead = true;
            break;
          }
          int page = t < a.seqs.pages_per_seq ? ptab[t] : -1;
          if (page < 0 || page >= a.pool_pages) {
            latch_status(a.status, kDevBounds);
            page = 0;
          }
          const uint8_t* src = reinterpret_cast<const uint8_t*>(a.pool) +
                               ((static_cast<size_t>(a.layer) * a.pool_pages + page) * nkv + it.kvh) * C::kRawUnit;
          mbar_arrive_expect_tx(&raw_full[r], C::kRawUnit);
          bulk_load(raw_ring + r * C::kRawUnit, src, C::kRawUnit, &raw_full[r]);
        }
      }
      // copies still in flight complete before shared memory is released
      for (int j = max(0, qu - RS); j < qu; ++j) mbar_wait(&raw_full[j % RS], (j / RS) & 1);
    }
  } else if (warp == 6) {
    // ---------------- L2 prefetch ----------------
    // Walks the same steps as the producer, at most kPrefetchSteps ahead of
    // it, and pulls their context pages into L2 with plain prefetches (one
    // 128-byte line per lane), so the producer's copies hit L2.
    int q = 0;
    bool stop = false;
    for (int rk = rec_begin; rk < rec_end && !stop; rk = next_rec(rk + 1)) {
      const Item it = decode(rk);
      const int slot = a.meta.slot[it.i], nctx = s_nctx[it.i];
      const int* ptab = a.seqs.page_table + static_cast<size_t>(slot) * a.seqs.pages_per_seq;
      for (int t0 = it.tb; t0 < it.te && !stop; t0 += 2, ++q) {
        if (s_issued + kPrefetchSteps <= q) {
          const unsigned long long w0 = global_ns();
          while (s_issued + kPrefetchSteps <= q) {
            if (abort_flag || global_ns() - w0 > kWaitLimitNs) {
              stop = true;
              break;
            }
            __nanosleep(200);
          }
          if (stop) break;
        }
        for (int u = 0; u < 2; ++u) {
          const int t = t0 + u;
          if (t >= it.te || t >= nctx || t >= a.seqs.pages_per_seq) continue;
          const int page = ptab[t];
          if (page < 0 || page >= a.pool_pages) continue;
          const size_t lp = static_cast<size_t>(a.layer) * a.pool_pages + page;
          const uint16_t* kp = a.pool + ((lp * 2 * nkv + it.kvh) * kKeyTile) * D;
          const uint16_t* vp = a.pool + (((lp * 2 + 1) * nkv + it.kvh) * D) * kKeyTile;
#pragma unroll
          for (int l = lane; l < kKeyTile * D * 2 / 128; l += 32) {   // 128-byte lines of a 64 x D tile
            asm volatile("prefetch.global.L2 [%0];" ::"l"(kp + l * 64));
            asm volatile("prefetch.global.L2 [%0];" ::"l"(vp + l * 64));
          }
        }
      }
    }
  } else {
    // ---------------- softmax / output warps ----------------
    const int quarter = warp & 3;                          // TMEM lanes 32*quarter .. +31
    const int half = SPREAD ? (lane >> 4) : 0;             // which unit of the step (SPREAD)
    const int row = SPREAD ? quarter * 16 + (lane & 15) : quarter * 32 + lane;   // query row r
    const bool active = (SPREAD ? quarter * 16 : quarter * 32) < R;              // warp-uniform
    const int jq = row / G;                                                     // block position of row r
    const uint32_t lane_tmem = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t o_tmem = lane_tmem + C::kOCol;
    const float sl2 = 1.4426950408889634f / sqrtf(static_cast<float>(D));   // log2(e)/sqrt(d)
    // waits taken by all 32 lanes together, so the warp-collective TMEM
    // accesses after them never diverge (also when a wait runs out)
    auto warp_wait = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, &abort_flag));
    };
    // Q rows of an item into TMEM (packed bf16 pairs): the thread's row,
    // all D dims (one thread per row) or D/2 dims (SPREAD, by half).
    auto load_q = [&](const Item& it) {
      if (active) {
        constexpr int kW = SPREAD ? D / 4 : D / 2;       // 32-bit words per thread
        uint32_t qv[kW];
        if (row < R) {
          const int j = row / G, g = row - j * G;
          const uint4* src = reinterpret_cast<const uint4*>(
              a.q + (static_cast<size_t>(it.i * B + j) * a.n_q_heads + it.kvh * G + g) * D + half * (D / 2));
#pragma unroll
          for (int c = 0; c < kW / 4; ++c) {
            const uint4 v4 = __ldcg(src + c);
            qv[4 * c] = v4.x;
            qv[4 * c + 1] = v4.y;
            qv[4 * c + 2] = v4.z;
            qv[4 * c + 3] = v4.w;
          }
        } else {
#pragma unroll
          for (int c = 0; c < kW; ++c) qv[c] = 0u;
        }
        if constexpr (SPREAD) {
          if constexpr (D == 128) tmem_st_half_u32<32>(lane_tmem + C::kQCol, qv);
          else tmem_st_half_u16<16>(lane_tmem + C::kQCol, qv);
        } else {
          if constexpr (D == 128) {
            uint32_t lo[32], hi[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              lo[c] = qv[c];
              hi[c] = qv[32 + c];
            }
            tmem_st_u32(lane_tmem + C::kQCol, lo);
            tmem_st_u32(lane_tmem + C::kQCol + 32, hi);
          } else {
            tmem_st_u32(lane_tmem + C::kQCol, qv);
          }
        }
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&q_ready);
    };
    // O row of this thread: D columns (one thread per row) or D/2 (SPREAD)
    auto o_scale = [&](float alpha) {
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
    // 64 S values of unit u (one thread per row) or of this thread's unit (SPREAD)
    auto load_s = [&](uint32_t s_tmem, int u, float (&sv)[64]) {
      if constexpr (SPREAD) tmem_ld_half64<64>(s_tmem, sv);
      else tmem_ld64(s_tmem + u * kKeyTile, sv);
    };
    auto mask = [&](float (&sv)[64], int nvalid) {
      if (nvalid < kKeyTile) {
#pragma unroll
        for (int c = 0; c < 64; ++c) sv[c] = c < nvalid ? sv[c] : -INFINITY;
      }
    };
    // p = 2^(s*sl2 - m), packed to bf16 pairs; returns the sum of p
    auto exp_pack = [&](const float (&sv)[64], float m, uint32_t (&pk)[32]) {
      float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float p0 = ex2(fmaf(sv[2 * c], sl2, -m));
        const float p1 = ex2(fmaf(sv[2 * c + 1], sl2, -m));
        s4[c & 3] += p0 + p1;
        pk[c] = Q8 ? pack_f16(p0, p1) : pack_bf16(p0, p1);
      }
      return (s4[0] + s4[1]) + (s4[2] + s4[3]);
    };
    int q = 0, k = 0;
    bool dead = false;
    grid_dep_wait();   // q comes from the projection kernel
    if (rec_begin < rec_end) load_q(decode(rec_begin));
    for (int rk = rec_begin; rk < rec_end && !dead; rk = next_rec(rk + 1), ++k) {
      const Item it = decode(rk);
      const int ns = (it.te - it.tb + 1) >> 1;
      const int len = s_len[it.i], nctx = s_nctx[it.i];
      // valid keys of unit t (0 if absent); causal: block position jq sees
      // the block's keys 0..jq (at least one, so a unit present is present
      // for every lane and the TMEM loads below stay warp-uniform)
      auto unit_valid = [&](int t) {
        return t >= it.te ? 0 : (t < nctx ? min(kKeyTile, len - t * kKeyTile) : (a.causal ? min(B, jq + 1) : B));
      };
      float m_run = -INFINITY, l_run = 0.f;   // l_run: this thread's share of the row sum
      for (int j = 0; j < ns; ++j) {
        const int qq = q + j, b = qq & 1;
        const uint32_t s_tmem = lane_tmem + b * C::kSCols;
        const int t0 = it.tb + 2 * j;
        const int n0 = unit_valid(t0), n1 = unit_valid(t0 + 1);
        if (!warp_wait(&s_full[b], (qq >> 1) & 1)) {
          give_up();
          dead = true;
          break;
        }
        tc_fence_after();
        if (active) {
          float sv[64];
          float mx;
          if constexpr (SPREAD) {
            load_s(s_tmem, 0, sv);
            mask(sv, half ? n1 : n0);
            mx = row_max(sv);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          } else {
            load_s(s_tmem, 0, sv);
            mask(sv, n0);
            mx = row_max(sv);
            if (n1 > 0) {
              load_s(s_tmem, 1, sv);
              mask(sv, n1);
              mx = fmaxf(mx, row_max(sv));
            }
          }
          mx *= sl2;   // log2 units
          if (j == 0) {
            m_run = mx;
          } else if (__any_sync(0xffffffffu, row < R && mx > m_run + kRescaleLog2)) {
            // O holds the products up to step qq-1: wait for them, then rescale
            if (!warp_wait(&kv_empty[(qq - 1) % S], ((qq - 1) / S) & 1)) {
              give_up();
              dead = true;
            }
            tc_fence_after();
            const float nm = fmaxf(m_run, mx);
            const float alpha = ex2(m_run - nm);
            l_run *= alpha;
            m_run = nm;
            if (!dead) o_scale(alpha);
          }
          uint32_t pk[32];
          if constexpr (SPREAD) {
            // sv still holds this thread's unit; P of unit `half` -> columns 32*half ..
            l_run += exp_pack(sv, m_run, pk);
            tmem_st_half_u32<32>(s_tmem, pk);
          } else {
            // P of unit 1 goes to columns 32..63, which still hold S of unit
            // 0: both units are read before either P is stored
            uint32_t pk1[32];
            if (n1 > 0) {   // sv holds unit 1
              l_run += exp_pack(sv, m_run, pk1);
              load_s(s_tmem, 0, sv);
              mask(sv, n0);
            }
            l_run += exp_pack(sv, m_run, pk);
            tmem_st_u32(s_tmem, pk);
            if (n1 > 0) tmem_st_u32(s_tmem + 32, pk1);
          }
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[b]);
        if (dead) break;
      }
      if (dead) break;
      // every S of this item has completed: Q's TMEM columns are free for the next item
      {
        const int rn = next_rec(rk + 1);
        if (rn < rec_end) load_q(decode(rn));
      }
      if (!warp_wait(&o_full, k & 1)) {
        give_up();
        break;
      }
      tc_fence_after();
      if (active) {
        if constexpr (SPREAD) l_run += __shfl_xor_sync(0xffffffffu, l_run, 16);
        const bool keep = row < R && it.slot < a.items_cap;
        float* po = a.part_o + (static_cast<size_t>(it.slot) * a.rows_pad + row) * D + half * (D / 2);
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
        if (keep && half == 0) a.part_ml[static_cast<size_t>(it.slot) * a.rows_pad + row] = make_float2(m_run, l_run);
        if (row == 0 && half == 0 && it.slot >= a.items_cap) latch_status(a.status, kDevBounds);   // host sizing prevents this
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&o_free);
      q += ns;
    }
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

// NC: chunk count up to which a row's partials are all loaded at once (the
// host's bound on the chunks per row picks the instantiation, so short rows
// do not pay registers, and occupancy, for 32 chunks); rows with more chunks
// take the general path.
template <int D, int NC>
__global__ void __launch_bounds__(32 * kCombineWarps) attn_combine_kernel(const __grid_constant__ AttnArgs a) {
  constexpr int kPer = D / 32;                 // dims per lane: 4 (D = 128) or 2 (D = 64)
  static_assert(NC >= 1 && NC <= 32, "one chunk per lane at most");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hq = blockIdx.x, i = blockIdx.y;
  const int j = blockIdx.z * kCombineWarps + warp;
  const int B = a.meta.B;
  const int nkv = a.n_kv_heads, G = a.n_q_heads / nkv;
  const int kvh = hq / G, gh = hq - kvh * G;
  // The lengths are final before any kernel of the pass starts (as for the
  // attention kernel's pages), so the row's chunk base is read before the
  // wait; the partials, written by the attention kernel, after it.
  int base = 0;
  for (int s = 0; s < i; ++s) base += nkv * seq_split(a, s).n_chunks;
  const int nch = seq_split(a, i).n_chunks;
  base += kvh * nch;
  grid_dep_wait();
  grid_dep_launch();
  if (j >= B || base + nch > a.items_cap) {
    if (j < B && lane == 0) latch_status(a.status, kDevBounds);
    return;
  }
  const int r = j * G + gh;
  const size_t rp = static_cast<size_t>(a.rows_pad);
  uint16_t* out = a.out + static_cast<size_t>(i * B + j) * a.n_q_heads * D + static_cast<size_t>(hq) * D + lane * kPer;
  if (nch <= NC) {
    // Every chunk in flight at once: lane c holds chunk c's (max, sum), and
    // every lane loads its dims of all partial rows before the weights are
    // known, so the merge costs about one memory latency.
    const float2 ml = lane < nch ? __ldcg(a.part_ml + (base + lane) * rp + r) : make_float2(-INFINITY, 0.f);
    const float* po = a.part_o + (static_cast<size_t>(base) * rp + r) * D + lane * kPer;
    float v[NC][kPer];
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      if (c < nch) {
        if constexpr (kPer == 4) {
          const float4 t = __ldcg(reinterpret_cast<const float4*>(po + c * rp * D));
          v[c][0] = t.x; v[c][1] = t.y; v[c][2] = t.z; v[c][3] = t.w;
        } else {
          const float2 t = __ldcg(reinterpret_cast<const float2*>(po + c * rp * D));
          v[c][0] = t.x; v[c][1] = t.y;
        }
      } else {
#pragma unroll
        for (int e = 0; e < kPer; ++e) v[c][e] = 0.f;
      }
    }
    float M = ml.x;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float w = lane < nch ? exp2f(ml.x - M) : 0.f;
    float L = w * ml.y;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    float acc[kPer];
#pragma unroll
    for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const float wc = __shfl_sync(0xffffffffu, w, c);
#pragma unroll
      for (int e = 0; e < kPer; ++e) acc[e] += wc * v[c][e];
    }
    const float inv = 1.f / L;
#pragma unroll
    for (int e = 0; e < kPer; ++e) out[e] = f32_to_bf16(acc[e] * inv);
    return;
  }
  float M = -INFINITY;
  for (int c = lane; c < nch; c += 32) M = fmaxf(M, a.part_ml[(base + c) * rp + r].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float L = 0.f;
  for (int c = lane; c < nch; c += 32) {
    const float2 ml = a.part_ml[(base + c) * rp + r];
    L += exp2f(ml.x - M) * ml.y;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  // chunk weights are recomputed from (max, sum) where they are used: one
  // broadcast load each
  const float* pm = &a.part_ml[static_cast<size_t>(base) * rp + r].x;
  float acc[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
  const float* po = a.part_o + (static_cast<size_t>(base) * rp + r) * D + lane * kPer;
  const size_t stride = rp * D;
  int c = 0;
  for (; c + 4 <= nch; c += 4) {
    float v[4][kPer], wv[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) wv[u] = exp2f(pm[(c + u) * 2 * rp] - M);
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
      for (int e = 0; e < kPer; ++e) acc[e] += wv[u] * v[u][e];
  }
  for (; c < nch; ++c) {
    const float wc = exp2f(pm[c * 2 * rp] - M);
#pragma unroll
    for (int e = 0; e < kPer; ++e) acc[e] += wc * __ldcg(po + c * stride + e);
  }
  const float inv = 1.f / L;
#pragma unroll
  for (int e = 0; e < kPer; ++e) out[e] = f32_to_bf16(acc[e] * inv);
}

template <int D, bool SPREAD, bool Q8>
cudaError_t launch_main(const AttnMaps& maps, const AttnArgs& a, const AttnSched& sched, int grid,
                        cudaStream_t stream) {
  using C = ACfg<D, Q8>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e =
        cudaFuncSetAttribute(attn_kernel<D, SPREAD, Q8>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_pdl(attn_kernel<D, SPREAD, Q8>, dim3(grid), dim3(attn_threads<Q8>()), C::kSmem, stream, maps, a,
                    sched);
}

template <int D>
cudaError_t launch_d(const AttnMaps& maps, const AttnArgs& a, const AttnSched& sched, int grid, int part,
                     cudaStream_t stream) {
  if (part == 0) {
    if (a.q8)
      return a.spread ? launch_main<D, true, true>(maps, a, sched, grid, stream)
                      : launch_main<D, false, true>(maps, a, sched, grid, stream);
    return a.spread ? launch_main<D, true, false>(maps, a, sched, grid, stream)
                    : launch_main<D, false, false>(maps, a, sched, grid, stream);
  }
  const dim3 grid_c(a.n_q_heads, a.meta.n_seq, (a.meta.B + kCombineWarps - 1) / kCombineWarps);
  const dim3 block_c(32 * kCombineWarps);
  if (a.max_chunks <= 8) return launch_pdl(attn_combine_kernel<D, 8>, grid_c, block_c, 0, stream, a);
  if (a.max_chunks <= 16) return launch_pdl(attn_combine_kernel<D, 16>, grid_c, block_c, 0, stream, a);
  return launch_pdl(attn_combine_kernel<D, 32>, grid_c, block_c, 0, stream, a);
}

}  // namespace

int attention_block_rows(int B) { return block_rows(B); }

int attention_ctas_per_sm(int head_dim, bool q8) {
  int n = 0;
  auto q = [&](auto kern, int smem, int threads) {
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, threads, smem) != cudaSuccess) n = 1;
  };
  if (q8) {
    if (head_dim == 128) q(attn_kernel<128, true, true>, ACfg<128, true>::kSmem, attn_threads<true>());
    else q(attn_kernel<64, true, true>, ACfg<64, true>::kSmem, attn_threads<true>());
  } else {
    if (head_dim == 128) q(attn_kernel<128, true, false>, ACfg<128>::kSmem, kThreads);
    else q(attn_kernel<64, true, false>, ACfg<64>::kSmem, kThreads);
  }
  return n < 1 ? 1 : n;
}

cudaError_t launch_attention(const AttnMaps& maps, const AttnArgs& a, const AttnSched& sched, int grid, int part,
                             cudaStream_t stream) {
  const int G = a.n_q_heads / a.n_kv_heads, R = G * a.meta.B;
  if (R > 128 || a.rows_pad < R) return cudaErrorInvalidValue;
  if (a.spread && R > 64) return cudaErrorInvalidValue;
  if (grid < 1 || grid > kSchedCtas || sched.off[grid] > kSchedItems) return cudaErrorInvalidValue;
  if (a.head_dim == 128) return launch_d<128>(maps, a, sched, grid, part, stream);
  if (a.head_dim == 64) return launch_d<64>(maps, a, sched, grid, part, stream);
  return cudaErrorInvalidValue;
}

}  // namespace dfl
