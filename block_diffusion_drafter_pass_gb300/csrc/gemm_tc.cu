// gemm_tc.cu - host side of the tensor-core GEMM: token-tile choice, the
// stream-K / data-parallel grid, and dispatch to the kernel instantiation of
// the epilogue's class (kernels in gemm_kernel.cuh, one translation unit per
// class: gemm_ec_*.cu).
#include "gemm_kernel.cuh"

namespace dfl {
using namespace gk;

namespace {
// CTA pairs over 256 x 256 pair tiles pay when every pair has one tile (the
// tile count fits one round) or the round-robin deal keeps at least half of
// the pairs' time busy: a pair MMA does twice the work per instruction, so
// even two uneven rounds beat a balanced single-CTA schedule.
bool pair_tiles_ok(int M, int N, int num_sms) {
  const long long nt = (N + kTileN - 1) / kTileN;
  if (nt < 2) return false;
  const long long pt = ((nt + 1) / 2) * ((M + 255) / 256), pairs = num_sms / 2;
  if (pt <= pairs) return true;
  const long long rounds = (pt + pairs - 1) / pairs;
  return static_cast<double>(pt) / static_cast<double>(rounds * pairs) >= 0.5;
}
}  // namespace

int gemm_token_tile(int M, int N, int num_sms) {
  if (M <= 16) return 16;
  if (M <= 32) return 32;
  if (M <= 64) return 64;
  if (M <= 128) return 128;
  const long long nt = (N + kTileN - 1) / kTileN;
  // 256-token tiles split over K between the two CTAs of a cluster whenever
  // two CTAs per tile fit in one wave: an MMA instruction of a 256-token tile
  // does twice the work of a 128-token one at the same issue cost, and the
  // split keeps the CTA count of 128-token tiles.
  if (2 * nt * ((M + 255) / 256) <= num_sms) return 256;
  // otherwise CTA pairs over 256-token tiles (two weight tiles per pair)
  if (pair_tiles_ok(M, N, num_sms)) return 256;
  // 256-token tiles, unless 128-token tiles keep clearly more SMs busy (a
  // tile count well under one wave)
  auto busy = [&](int bn) {
    const long long t = nt * ((M + bn - 1) / bn);
    const long long waves = (t + num_sms - 1) / num_sms;
    return static_cast<double>(t) / static_cast<double>(waves * num_sms);
  };
  return busy(128) > busy(256) + 0.05 ? 128 : 256;
}

namespace {
// Clusters of two CTA pairs, each over half of the k-blocks of one pair tile,
// when four CTAs per pair tile fit one wave (256-token tiles).
bool pair_split_ok(int M, int N, int K, int num_sms) {
  const long long nt = (N + kTileN - 1) / kTileN;
  if (M <= 128 || nt < 2 || (K + kTileK - 1) / kTileK < 2) return false;
  return 4 * ((nt + 1) / 2) * ((M + 255) / 256) <= num_sms;
}
}  // namespace

int gemm_pair_mode(int M, int N, int K, int splits, int num_sms) {
  if (splits != 0 || M <= 128 || K < 1) return 0;
  if (pair_split_ok(M, N, K, num_sms)) return 2;
  const long long nt = (N + kTileN - 1) / kTileN;
  const long long tiles = nt * ((M + 255) / 256);
  if (2 * tiles <= num_sms && (K + kTileK - 1) / kTileK >= 2) return 0;   // single-CTA cluster split
  if (!pair_tiles_ok(M, N, num_sms)) return 0;
  // Round-robin pairs leave (rounds x pairs - pair tiles) pair slots idle.
  // Stream-K over the pairs gives every pair the same MMA work, but each
  // split tile costs a partial tile written by one CTA and read back by the
  // finishing one (about as long as the epilogue itself), so it is taken only
  // when round-robin would keep under 60% of the pairs busy (one full round
  // and a short second one: the fused K/V projection of 5 layers at 512
  // tokens).
  const long long pt = ((nt + 1) / 2) * ((M + 255) / 256), pairs = num_sms / 2;
  const long long rounds = (pt + pairs - 1) / pairs;
  return rounds > 1 && static_cast<double>(pt) / static_cast<double>(rounds * pairs) < 0.6 ? 3 : 1;
}

bool gemm_cluster_split(int M, int N, int K, int splits, int num_sms) {
  if (splits != 0 || gemm_token_tile(M, N, num_sms) != 256 || pair_split_ok(M, N, K, num_sms)) return false;
  const long long tiles = static_cast<long long>((N + kTileN - 1) / kTileN) * ((M + 255) / 256);
  return 2 * tiles <= num_sms && (K + kTileK - 1) / kTileK >= 2;
}

int gemm_act_rows(int M, int N, int K, int num_sms) {
  const int BN = gemm_token_tile(M, N, num_sms);
  return gemm_pair_mode(M, N, K, 0, num_sms) ? BN / 2 : BN;
}

int gemm_grid(int M, int N, int K, int splits, size_t partial_elems, int num_sms) {
  const int BN = gemm_token_tile(M, N, num_sms);
  const long long tiles = static_cast<long long>((N + kTileN - 1) / kTileN) * ((M + BN - 1) / BN);
  const int kb = (K + kTileK - 1) / kTileK;
  // one cluster of two CTAs per tile, each with half of the k-blocks: the
  // stream-K partition of 2 x tiles CTAs is exactly that split
  if (gemm_cluster_split(M, N, K, splits, num_sms)) return static_cast<int>(2 * tiles);
  // CTA pairs take whole pair tiles round-robin; split pairs one pair tile
  // per cluster of four
  if (const int pm = gemm_pair_mode(M, N, K, splits, num_sms)) {
    const long long pair_tiles = static_cast<long long>(((N + kTileN - 1) / kTileN + 1) / 2) * ((M + BN - 1) / BN);
    if (pm == 2) return static_cast<int>(4 * pair_tiles);
    // stream-K pairs need two 128 x 256 partial slots per CTA; without room
    // for them the pairs take whole tiles round-robin
    if (pm == 3 && static_cast<long long>(num_sms / 2) * 2 * 2 * kTileN * BN <= static_cast<long long>(partial_elems))
      return static_cast<int>(2 * std::min<long long>(pair_tiles * kb, num_sms / 2));
    return static_cast<int>(2 * std::min<long long>(pair_tiles, num_sms / 2));
  }
  const long long units = tiles * kb;
  long long G = splits > 0 ? tiles * std::min(splits, kb) : num_sms;
  // Tensor-bound tiles (BN >= 128) that fit in one wave: one whole tile per
  // CTA. Splitting them would buy idle SMs at the price of partial tiles the
  // finishing CTA must read back while the other CTAs' operand streams load
  // the memory system.
  if (splits == 0 && BN >= 128 && tiles <= num_sms) G = tiles;
  if (G > units) G = units;
  // 2 partial slots of 128 x BN floats per CTA, unless every CTA owns whole
  // tiles: the largest grid up to G that either divides the tile count (no
  // partials) or fits the partial buffer
  const long long cap = static_cast<long long>(partial_elems / (2ull * kTileN * BN));
  if (G > cap && tiles % G != 0) {
    long long d = std::min<long long>(G, tiles);
    while (d > cap && tiles % d != 0) --d;
    G = d;
  }
  return static_cast<int>(std::max<long long>(G, 1));
}

cudaError_t launch_gemm(const AMaps& amaps, const ARegions& regions, const CUtensorMap& xmap, int M, int N, int K,
                        int splits, const GemmEpi& epi, const GemmWork& work, int num_sms, cudaStream_t stream) {
  if (M <= 0) return cudaSuccess;
  if (regions.pair != 32 && regions.pair != 64) return cudaErrorInvalidValue;
  const int BN = gemm_token_tile(M, N, num_sms);
  GemmArgs a{};
  a.M = M;
  a.N = N;
  a.K = K;
  a.k_blocks = (K + kTileK - 1) / kTileK;
  a.n_tiles = (N + kTileN - 1) / kTileN;
  a.m_tiles = (M + BN - 1) / BN;
  a.units = static_cast<long long>(a.n_tiles) * a.m_tiles * a.k_blocks;
  a.grid = gemm_grid(M, N, K, splits, work.partial_elems, num_sms);
  a.csplit = gemm_cluster_split(M, N, K, splits, num_sms) ? 1 : 0;
  a.pair = gemm_pair_mode(M, N, K, splits, num_sms);
  a.workers = a.grid;
  if (a.pair == 3) {
    const long long tiles = static_cast<long long>(a.n_tiles) * a.m_tiles;
    const long long pair_tiles = static_cast<long long>((a.n_tiles + 1) / 2) * a.m_tiles;
    const bool room = static_cast<size_t>(a.grid) * 2 * kTileN * BN <= work.partial_elems && tiles <= work.n_tickets;
    if (room) {
      a.workers = a.grid / 2;
      a.units = pair_tiles * a.k_blocks;
    } else {
      a.pair = 1;   // gemm_grid chose the round-robin grid for this case
    }
  }
  // the pair exchange addresses a 128 x 128 float block of the peer's ring
  // (BN = 256) and pairs CTAs 2t, 2t + 1
  if (a.csplit && (BN != 256 || a.grid != 2 * a.n_tiles * a.m_tiles)) return cudaErrorInvalidValue;
  a.status = epi.status;
  a.partial = work.partial;
  a.tickets = work.tickets;
  if (!a.pair && static_cast<long long>(a.n_tiles) * a.m_tiles > work.n_tickets &&
      a.grid % (a.n_tiles * a.m_tiles) != 0)
    return cudaErrorInvalidValue;
  switch (epilogue_class(epi.kind)) {
    case kEcNorm: return launch_ec_norm(amaps, regions, xmap, a, epi, BN, stream);
    case kEcRope: return launch_ec_rope(amaps, regions, xmap, a, epi, BN, stream);
    case kEcSwiglu: return launch_ec_swiglu(amaps, regions, xmap, a, epi, BN, stream);
    case kEcArgmax: return launch_ec_argmax(amaps, regions, xmap, a, epi, BN, stream);
    default: return launch_ec_f32(amaps, regions, xmap, a, epi, BN, stream);
  }
}

}  // namespace dfl
