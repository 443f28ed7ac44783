// noalloc.cu - a GEMM entry point that never allocates device memory.
//
// dflash_debug_gemm allocates its split-K workspace with cudaMalloc on every
// call. Some callers cannot do that: cudaMalloc and cudaFree may synchronise
// the device, which a latency-critical loop must avoid; a caching allocator
// (PyTorch's, for one) may already hold all free memory; and while another
// thread of the process has a stream capture in progress in global mode,
// cudaMalloc is an unsafe call. dflash_gemm_noalloc serves them: its split-K
// partials, tile tickets and status word live in one file-scope device array
// of fixed size, which every GPU that loads this library keeps until the
// process exits. The caller still provides W, X and Y.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "dflash.h"
#include "internal.h"

namespace {

using namespace dfl;

// Scratch layout: [kPartialFloats floats of split-K partials][kTickets ints][1 status int].
constexpr size_t kPartialFloats = size_t(2) << 20;   // 8 MiB of fp32 partials
constexpr int kTickets = 4096;
constexpr size_t kScratchBytes = kPartialFloats * sizeof(float) + (kTickets + 1) * sizeof(int);

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

// Device address of the scratch array on the current device, looked up once
// per device. In host code the array's name only stands for the symbol; the
// device address must come from cudaGetSymbolAddress.
cudaError_t scratch_on_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" dflash_status dflash_gemm_noalloc(const uint16_t* W, const uint16_t* X, float* Y, int N, int M, int K,
                                             int splits, void* stream_v) {
  if (!W || !X || !Y || N < 1 || M < 1 || K < 8 || K % 8 || splits < 0) {
    set_unattached_error("dflash_gemm_noalloc: null pointer or bad shape (K must be a positive multiple of 8)");
    return DFLASH_EINVAL;
  }
  if ((reinterpret_cast<uintptr_t>(W) | reinterpret_cast<uintptr_t>(X)) & 15) {
    set_unattached_error("dflash_gemm_noalloc: W and X must be 16-byte aligned");
    return DFLASH_EINVAL;
  }
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    set_unattached_error("dflash_gemm_noalloc: no CUDA device");
    return DFLASH_ECUDA;
  }
  const int BN = gemm_token_tile(M, N, sms);
  const long long tiles = static_cast<long long>(ceil_div(M, BN)) * ceil_div(N, 128);
  const int k_blocks = ceil_div(K, 64);
  if (tiles > kTickets) {
    set_unattached_error("dflash_gemm_noalloc: more than 4096 output tiles of 128 x 16..256");
    return DFLASH_EINVAL;
  }
  if (splits > 0) {
    // An explicit split factor s runs tiles x min(s, k_blocks) CTAs. With one
    // split per tile every CTA owns a whole tile and writes no partials; with
    // more, each CTA has two 128 x BN partial slots.
    const int per_tile = std::min(splits, k_blocks);
    const long long need = 2 * tiles * per_tile * 128 * BN;
    if (per_tile > 1 && need > static_cast<long long>(kPartialFloats)) {
      set_unattached_error("dflash_gemm_noalloc: split-K partials exceed the fixed 8 MiB scratch "
                           "(2 x splits x M rounded up to the token tile x roundup(N,128) floats); use fewer splits");
      return DFLASH_EINVAL;
    }
  }
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  void* base = nullptr;
  cudaError_t e = scratch_on_current_device(&base);
  if (e != cudaSuccess) {
    set_unattached_error("dflash_gemm_noalloc: cudaGetSymbolAddress of the scratch array failed");
    return DFLASH_ECUDA;
  }
  AMaps am;
  CUtensorMap xm;
  const int xbox = splits == 0 ? gemm_act_rows(M, N, K, sms) : BN;   // CTA pairs each load half the tokens
  if (!encode_matrix_map(&am.m[0], W, N, K, kWeightBoxRows) || !encode_matrix_map(&xm, X, M, K, xbox)) {
    set_unattached_error("dflash_gemm_noalloc: cannot describe W or X for TMA");
    return DFLASH_EINVAL;
  }
  GemmWork work;
  work.partial = reinterpret_cast<float*>(base);
  work.partial_elems = kPartialFloats;
  work.tickets = reinterpret_cast<int*>(reinterpret_cast<unsigned char*>(base) + kPartialFloats * sizeof(float));
  work.n_tickets = kTickets;
  int* status = work.tickets + kTickets;
  // Tickets and the status word must start at zero; the previous call's
  // contents are still there.
  if (cudaMemsetAsync(work.tickets, 0, (kTickets + 1) * sizeof(int), stream) != cudaSuccess) {
    set_unattached_error("dflash_gemm_noalloc: clearing the scratch tickets failed");
    return DFLASH_ECUDA;
  }
  GemmEpi ep;
  std::memset(&ep, 0, sizeof(ep));
  ep.kind = EPI_F32_STORE;
  ep.out_f32 = Y;
  ep.ld_out = N;
  ep.status = status;
  ARegions rg;
  std::memset(&rg, 0, sizeof(rg));
  rg.n_regions = 1;
  rg.pair = 64;
  rg.tile_begin[1] = ceil_div(N, 128);
  if (launch_gemm(am, rg, xm, M, N, K, splits, ep, work, sms, stream) != cudaSuccess) {
    set_unattached_error("dflash_gemm_noalloc: kernel launch failed");
    return DFLASH_ECUDA;
  }
  // The status word is read on the caller's stream, never on the legacy
  // default stream: a blocking copy there would wait for every blocking
  // stream of the device and would break another thread's global-mode capture.
  int st = 0;
  if (cudaMemcpyAsync(&st, status, sizeof(int), cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess) {
    set_unattached_error("dflash_gemm_noalloc: CUDA error while waiting for the GEMM");
    return DFLASH_ECUDA;
  }
  if (st & kDevTimeout) return DFLASH_ETIMEOUT;
  if (st) return DFLASH_EDEVICE;
  return DFLASH_OK;
}
