// gemv_host.cu -- per-shape configuration and launch of the N=1 kernels.
//
// The configuration table follows the source page's rule "pick by (M, K)
// microbench" ("Decode V2 -- resident executor", section 6): the page packs
// NR = 4 rows per block for M >= 4096 and keeps one row for M = 2048 on a
// 70-SM desktop part.  Here the equivalents are the row-group width G (threads
// sharing one row, set by K), the batch RB (rows in flight per thread) and the
// number of groups per block, with the grid sized to fill all SMs once
// (persistent blocks, each owning a contiguous range of rows).
#include <algorithm>
#include <cstdlib>
#include <map>
#include <mutex>
#include <tuple>

#include "gemv_dispatch.cuh"
#include "gemv_tma_dispatch.cuh"

namespace nf4k {

namespace {

const void* kernel_ptr(int epi, int nch, int rb, bool big, bool xb) {
  switch (epi) {
    case EPI_PLAIN: return GemvDispatch<EPI_PLAIN>::ptr(nch, rb, big, xb);
    case EPI_RESID: return GemvDispatch<EPI_RESID>::ptr(nch, rb, big, xb);
    case EPI_SWIGLU: return GemvDispatch<EPI_SWIGLU>::ptr(nch, rb, big, xb);
    case EPI_QKV: return GemvDispatch<EPI_QKV>::ptr(nch, rb, big, xb);
    case EPI_GLU: return GemvDispatch<EPI_GLU>::ptr(nch, rb, big, xb);
    default: return GemvDispatch<EPI_ARGMAX>::ptr(nch, rb, big, xb);
  }
}

// Largest block the instantiation can launch (its register use decides).
int max_threads(int epi, int nch, int rb, bool big) {
  int m = 1 << 30;
  for (int xb = 0; xb < 2; ++xb) {
    cudaFuncAttributes attr{};
    if (cudaFuncGetAttributes(&attr, kernel_ptr(epi, nch, rb, big, xb != 0)) != cudaSuccess) return 0;
    m = attr.maxThreadsPerBlock < m ? attr.maxThreadsPerBlock : m;
  }
  return m;
}

int env_int(const char* name, int dflt) {
  const char* v = std::getenv(name);
  return (v && *v) ? std::atoi(v) : dflt;
}

struct Key {
  int epi, device;
  int64_t M, K;
  bool operator<(const Key& o) const {
    return std::tie(epi, device, M, K) < std::tie(o.epi, o.device, o.M, o.K);
  }
};

std::mutex g_mu;
std::map<Key, GemvConfig> g_cache;
std::map<Key, TmaConfig> g_tma_cache;

const void* tma_ptr(int epi, int nch, int rb, int sub, bool xb, int lut) {
  switch (epi) {
    case EPI_PLAIN: return GemvTmaDispatch<EPI_PLAIN>::ptr(nch, rb, sub, xb, lut);
    case EPI_RESID: return GemvTmaDispatch<EPI_RESID>::ptr(nch, rb, sub, xb, lut);
    case EPI_SWIGLU: return GemvTmaDispatch<EPI_SWIGLU>::ptr(nch, rb, sub, xb, lut);
    case EPI_QKV: return GemvTmaDispatch<EPI_QKV>::ptr(nch, rb, sub, xb, lut);
    case EPI_GLU: return GemvTmaDispatch<EPI_GLU>::ptr(nch, rb, sub, xb, lut);
    default: return GemvTmaDispatch<EPI_ARGMAX>::ptr(nch, rb, sub, xb, lut);
  }
}

}  // namespace

GemvConfig choose_gemv_config(int epi, int64_t M, int64_t K, int device) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_cache.find(Key{epi, device, M, K});
    if (it != g_cache.end()) return it->second;
  }
  GemvConfig c{};
  const bool two = (epi == EPI_SWIGLU);
  const int H = (int)(K / 32);            // 16-byte code chunks per row
  const int G1 = 32 * ((H + 31) / 32);    // group width with one chunk per thread
  const int G2 = 32 * ((H + 63) / 64);    // group width with two chunks per thread
  // candidates in order of preference: (nch, rb, big)
  const int cand[][3] = {
      {H <= 32 ? 1 : (H <= 64 ? 2 : 1), two ? 2 : 4, 0},
      {1, 2, 0}, {2, 2, 0}, {1, 2, 1}, {2, 2, 1}};
  int pick = -1, mt = 0;
  for (int i = 0; i < 5 && pick < 0; ++i) {
    int nch = cand[i][0], rb = cand[i][1];
    const bool big = cand[i][2] != 0;
    if (i == 0) rb = env_int("NF4_GEMV_RB", rb);
    if (!gemv_variant_exists(nch, rb, big)) continue;
    const int G = (H <= 32) ? 32 : (nch == 1 ? G1 : G2);
    const int m = max_threads(epi, nch, rb, big);
    if (G <= m && G <= 1024) {
      pick = i;
      c.nch = nch;
      c.rb = rb;
      c.big = big;
      c.G = G;
      mt = m;
    }
  }
  if (pick < 0) {  // cannot happen for K <= 65536: (2, 2, big) needs G2 <= 1024
    c.blocks = 0;
    return c;
  }
  int gpc = mt / c.G;
  gpc = gpc < 1 ? 1 : gpc;
  const int gpc_cap = (c.G == 32) ? 32 : 15;  // named barrier ids 1..15
  gpc = gpc > gpc_cap ? gpc_cap : gpc;
  gpc = env_int("NF4_GEMV_GPC", gpc);
  if (gpc * c.G > mt) gpc = mt / c.G;
  if (gpc > gpc_cap) gpc = gpc_cap;
  if (gpc < 1) gpc = 1;
  const int nv = two ? 2 : 1;
  c.gpc = gpc;
  c.smem = LUT_BYTES + gpc * 2 * nv * c.rb * (c.G / 32) * (int)sizeof(float);

  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
  for (int xb = 0; xb < 2; ++xb)
    cudaFuncSetAttribute(kernel_ptr(epi, c.nch, c.rb, c.big, xb != 0), cudaFuncAttributeMaxDynamicSharedMemorySize,
                         c.smem);
  int bps = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, kernel_ptr(epi, c.nch, c.rb, c.big, true), c.G * c.gpc,
                                                c.smem);
  bps = bps < 1 ? 1 : bps;
  bps = env_int("NF4_GEMV_BPS", bps);
  const int64_t want = (M + c.gpc - 1) / c.gpc;
  const int64_t have = (int64_t)(sms > 0 ? sms : 1) * bps;
  c.blocks = (int)(want < have ? want : have);
  cudaGetLastError();  // attribute queries leave no sticky state behind
  std::lock_guard<std::mutex> lk(g_mu);
  g_cache[Key{epi, device, M, K}] = c;
  return c;
}

// Groups of G threads per block for the bulk-copy kernel, from a cost model
// of the busiest group: blocks take ceil(M / blocks) rows each, in stages of
// GPS x RB rows handed round robin to the gpc / GPS sets of groups, and a
// block's groups share the SM's arithmetic, so the block's time goes as
// (stages of the busiest set) x RB x gpc.  Blocks keep at least 8 compute
// warps; ties go to the count nearest 768 compute threads.  (Measured on
// 13824 x 5120: 4 groups of 160 threads, 2 per stage, 12.3 us; 5 groups, 1 per
// stage, whose last stages leave three groups idle, 13.4 us.)
int tma_groups_per_stage(int gpc, int G, int rb, int nv, int64_t K, const cudaFuncAttributes& attr, int device);

int pick_groups(int G, int rb, int nv, int64_t M, int64_t K, const cudaFuncAttributes& attr, int device) {
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
  sms = sms > 0 ? sms : 1;
  const int max_threads = attr.maxThreadsPerBlock < 1024 ? attr.maxThreadsPerBlock : 1024;
  int gcap = (max_threads - 32) / G;
  gcap = gcap > 14 ? 14 : gcap;
  if (gcap < 1) return 0;
  int gmin = (256 + G - 1) / G;
  gmin = gmin > gcap ? gcap : gmin;
  int64_t cost[15] = {0};
  int64_t min_cost = -1;
  for (int g = gmin; g <= gcap; ++g) {
    const int d = tma_groups_per_stage(g, G, rb, nv, K, attr, device);
    const int64_t SR = (int64_t)d * rb;
    const int64_t blocks = std::min<int64_t>((M + SR - 1) / SR, sms);
    const int64_t rows = (M + blocks - 1) / blocks;
    const int64_t n_it = (rows + SR - 1) / SR;
    const int64_t sets = g / d;
    cost[g] = ((n_it + sets - 1) / sets) * rb * g;
    if (min_cost < 0 || cost[g] < min_cost) min_cost = cost[g];
  }
  // within 2% of the cheapest counts as a tie
  int best = 0;
  for (int g = gmin; g <= gcap; ++g)
    if (cost[g] * 50 <= min_cost * 51 && (best == 0 || std::abs(g * G - 768) < std::abs(best * G - 768))) best = g;
  return best;
}

// Groups per stage: the largest divisor of gpc whose stages still fit twice
// beside the pair table and the reduction slots (big block-wide stages stream
// best; long rows need small ones).
int tma_groups_per_stage(int gpc, int G, int rb, int nv, int64_t K, const cudaFuncAttributes& attr, int device) {
  int optin = 0;
  cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
  const int red_set = gpc * (nv * rb * (G / 32) * (int)sizeof(float) + (int)sizeof(int));
  const int avail = optin - (int)attr.sharedSizeBytes - LUT_BYTES - red_set - 256;
  const int one_group = nv * rb * (int)(K / 2 + K / 16);
  for (int d = gpc; d >= 1; --d)
    if (gpc % d == 0 && 2 * d * one_group <= avail) return d;
  return 1;
}

// Bulk-copy kernel: x-stationary row groups as in the register kernel, plus a
// producer warp and a ring of S stages of SR rows each, one block per SM.
TmaConfig choose_tma_config(int epi, bool x_bf16, int64_t M, int64_t K, int device) {
  const int key_epi = 2 * epi + (x_bf16 ? 1 : 0);
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_tma_cache.find(Key{key_epi, device, M, K});
    if (it != g_tma_cache.end()) return it->second;
  }
  TmaConfig c{};
  c.ok = false;
  const bool two = (epi == EPI_SWIGLU);
  const int nv = two ? 2 : 1;
  const int H = (int)(K / 32);
  if (K % 256 != 0) return c;  // scale rows must be whole 16-byte units for the bulk copies
  if (H <= 32) {
    c.nch = 1;
    c.G = 32;
  } else if (H <= 64) {
    // one warp per row, two chunks per thread (no cross-warp reduction), or
    // for many rows of one matrix two warps per row, one chunk per thread
    // (more warps to hide the pair-table loads; measured with fp32 levels:
    // 151936 x 2048 48.5 against 49.7 us, 22016 x 2048 interleaved gate/up
    // 11.0 against 12.2 us; the two-matrix SwiGLU keeps two chunks, 10.6
    // against 12.0 us)
    const bool many_rows = M >= 16384 && epi != EPI_SWIGLU;
    c.nch = env_int("NF4_TMA_NCH", many_rows ? 1 : 2);
    c.G = c.nch == 2 ? 32 : 64;
  } else if (32 * ((H + 31) / 32) <= 992 && env_int("NF4_TMA_NCH", 1) == 1) {
    c.nch = 1;
    c.G = 32 * ((H + 31) / 32);
  } else {
    c.nch = 2;
    c.G = 32 * ((H + 63) / 64);
  }
  // rows per group and stage: 8 for one-chunk shapes (long per-warp work
  // amortizes the per-stage reduction; measured best for 2048 x 11008 and
  // 13824 x 5120), else 4; fewer when two stages would not fit beside the
  // pair table
  c.rb = c.nch == 1 ? 8 : 4;
  while (c.rb > 2 && 2 * c.rb * nv * (int)(K / 2 + K / 16) > 150 * 1024) c.rb /= 2;
  // two chunks per thread and few rows (short kernels): 2 rows per stage start
  // the computation sooner (measured with fp32 levels: 2048 x 2048 3.48
  // against 3.44 us, the fused 3B q/k/v 3.95 against 4.14, 256 x 2048 2.68
  // against 3.33; SwiGLU's 11008 rows are faster with 4: 10.6 against 11.2)
  if (c.nch == 2 && M < 4096) c.rb = 2;
  c.rb = env_int("NF4_TMA_RB", c.rb);
  // every activation dtype uses the exact fp32 levels; NF4_LUT=1 opts bf16
  // activations into the narrower fp16-level mixed-precision loop
  c.lut = env_int("NF4_LUT", LUT_F32) == LUT_F16MIX ? LUT_F16MIX : LUT_F32;
  auto lut_for = [&](int xb) { return xb ? c.lut : (int)LUT_F32; };
  // each activation dtype has its own instance and configuration (their
  // register use differs); when a row group does not fit in one block, retry
  // with fewer rows per stage
  const int xb = x_bf16 ? 1 : 0;
  cudaFuncAttributes attr{};
  const void* fn = nullptr;
  int gpc = 1;
  for (int attempt = 0;; ++attempt) {
    // rows per full barrier within a group's rows: all of them unless asked
    c.sub = env_int("NF4_TMA_SUB", c.rb);
    if (!gemv_tma_variant_exists(c.nch, c.rb, c.sub)) c.sub = c.rb;
    if (!gemv_tma_variant_exists(c.nch, c.rb, c.sub)) return c;
    fn = tma_ptr(epi, c.nch, c.rb, c.sub, x_bf16, lut_for(xb));
    if (fn == nullptr || cudaFuncGetAttributes(&attr, fn) != cudaSuccess) {
      cudaGetLastError();
      return c;
    }
    const int env_threads = env_int("NF4_TMA_THREADS", 0);
    if (env_threads > 0) {
      gpc = (env_threads + c.G / 2) / c.G;
      gpc = gpc < 1 ? 1 : (gpc > 14 ? 14 : gpc);
      while (gpc > 1 && gpc * c.G + 32 > attr.maxThreadsPerBlock) --gpc;
    } else {
      gpc = pick_groups(c.G, c.rb, nv, M, K, attr, device);
    }
    if (gpc >= 1 && gpc * c.G + 32 <= attr.maxThreadsPerBlock) break;
    if (c.rb == 2 || attempt > 2) return c;
    c.rb /= 2;
  }
  c.gpc = gpc;
  c.threads = gpc * c.G + 32;
  const int row_bytes = (int)(K / 2), srow_bytes = (int)(K / 16);
  // per stage: the stage itself, its two barriers, and one reduction slot
  // (NV x RB x warps-per-group partial sums) plus a counter per group; one
  // extra slot set on top (S + 1 slots)
  const int red_set = gpc * (nv * c.rb * (c.G / 32) * (int)sizeof(float) + (int)sizeof(int));
  int optin = 0;
  cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
  const int max_stages = 32;
  const int avail = optin - (int)attr.sharedSizeBytes - LUT_BYTES - red_set - 256;
  const int one_group = nv * c.rb * (row_bytes + srow_bytes);
  int gps = tma_groups_per_stage(gpc, c.G, c.rb, nv, K, attr, device);
  const int gps_env = env_int("NF4_TMA_GPS", 0);
  if (gps_env > 0 && gpc % gps_env == 0 && 2 * gps_env * one_group <= avail) gps = gps_env;
  c.GPS = gps;
  c.SR = gps * c.rb;
  // When every group gets a single stage (few rows per block, long rows),
  // split its rows over two full barriers so it can start on the first half
  // while the second is in flight (measured on 2048 x 11008: 6.6 us against
  // 6.9 us; with several stages per group the split costs more than it saves)
  if (env_int("NF4_TMA_SUB", 0) == 0 && c.rb >= 4 && gemv_tma_variant_exists(c.nch, c.rb, c.rb / 2)) {
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    const int64_t blocks_est = std::min<int64_t>((M + c.SR - 1) / c.SR, sms > 0 ? sms : 1);
    const int64_t rows_pb = (M + blocks_est - 1) / blocks_est;
    const int64_t per_group = ((rows_pb + c.SR - 1) / c.SR + (gpc / gps) - 1) / (gpc / gps);
    const void* half = tma_ptr(epi, c.nch, c.rb, c.rb / 2, x_bf16, lut_for(xb));
    cudaFuncAttributes ah{};
    if (per_group <= 1 && half != nullptr && cudaFuncGetAttributes(&ah, half) == cudaSuccess &&
        ah.maxThreadsPerBlock >= c.threads && ah.sharedSizeBytes == attr.sharedSizeBytes) {
      c.sub = c.rb / 2;
      fn = half;
    }
    cudaGetLastError();
  }
  // rows per full barrier: SUB when a group's rows are split (the consumers
  // start on the first rows of a stage while the rest are in flight), else
  // one barrier for the whole stage
  c.subr = c.sub < c.rb ? c.sub : c.SR;
  c.nb = c.SR / c.subr;
  const int bars_bytes = 8 * (c.nb + 1);  // per stage
  c.codes_bytes = c.SR * row_bytes;
  c.scales_bytes = c.SR * srow_bytes;
  c.stage_bytes = nv * (c.codes_bytes + c.scales_bytes);
  int S = (avail - 16) / (c.stage_bytes + bars_bytes + red_set);
  const int cap = env_int("NF4_TMA_STAGES", max_stages);
  S = S > cap ? cap : S;
  S = S > max_stages ? max_stages : S;
  if (S < 2) return c;
  c.S = S;
  c.bar_off = LUT_BYTES + S * c.stage_bytes;
  c.red_off = (c.bar_off + bars_bytes * S + 15) / 16 * 16;
  c.smem = c.red_off + (S + 1) * red_set;
  cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, c.smem);
  int sms = 0, bps = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, fn, c.threads, c.smem);
  if (bps < 1) {
    cudaGetLastError();
    return c;
  }
  const int64_t want = (M + c.SR - 1) / c.SR;
  const int64_t have = (int64_t)sms * bps;
  c.blocks = (int)(want < have ? want : have);
  c.ok = true;
  cudaGetLastError();
  std::lock_guard<std::mutex> lk(g_mu);
  g_tma_cache[Key{key_epi, device, M, K}] = c;
  return c;
}

cudaError_t launch_gemv_tma(int epi, bool xb, const GemvArgs& a, const TmaConfig& c, cudaStream_t s) {
  TmaPlan p{c.SR, c.GPS, c.S, c.stage_bytes, c.codes_bytes, c.scales_bytes, c.bar_off, c.red_off, c.subr, c.nb};
  switch (epi) {
    case EPI_PLAIN:
      return GemvTmaDispatch<EPI_PLAIN>::launch(c.nch, c.rb, c.sub, xb, xb ? c.lut : (int)LUT_F32, a, p, c.blocks, c.threads, c.smem, s);
    case EPI_RESID:
      return GemvTmaDispatch<EPI_RESID>::launch(c.nch, c.rb, c.sub, xb, xb ? c.lut : (int)LUT_F32, a, p, c.blocks, c.threads, c.smem, s);
    case EPI_SWIGLU:
      return GemvTmaDispatch<EPI_SWIGLU>::launch(c.nch, c.rb, c.sub, xb, xb ? c.lut : (int)LUT_F32, a, p, c.blocks, c.threads, c.smem, s);
    case EPI_QKV:
      return GemvTmaDispatch<EPI_QKV>::launch(c.nch, c.rb, c.sub, xb, xb ? c.lut : (int)LUT_F32, a, p, c.blocks, c.threads, c.smem, s);
    case EPI_GLU:
      return GemvTmaDispatch<EPI_GLU>::launch(c.nch, c.rb, c.sub, xb, xb ? c.lut : (int)LUT_F32, a, p, c.blocks, c.threads, c.smem, s);
    default:
      return GemvTmaDispatch<EPI_ARGMAX>::launch(c.nch, c.rb, c.sub, xb, xb ? c.lut : (int)LUT_F32, a, p, c.blocks, c.threads, c.smem, s);
  }
}

cudaError_t launch_gemv(int epi, bool xb, const GemvArgs& a, GemvConfig cfg, cudaStream_t s) {
  if (cfg.blocks < 1) return cudaErrorInvalidConfiguration;
  switch (epi) {
    case EPI_PLAIN: return GemvDispatch<EPI_PLAIN>::launch(cfg.nch, cfg.rb, cfg.big, xb, a, cfg, s);
    case EPI_RESID: return GemvDispatch<EPI_RESID>::launch(cfg.nch, cfg.rb, cfg.big, xb, a, cfg, s);
    case EPI_SWIGLU: return GemvDispatch<EPI_SWIGLU>::launch(cfg.nch, cfg.rb, cfg.big, xb, a, cfg, s);
    case EPI_QKV: return GemvDispatch<EPI_QKV>::launch(cfg.nch, cfg.rb, cfg.big, xb, a, cfg, s);
    case EPI_GLU: return GemvDispatch<EPI_GLU>::launch(cfg.nch, cfg.rb, cfg.big, xb, a, cfg, s);
    default: return GemvDispatch<EPI_ARGMAX>::launch(cfg.nch, cfg.rb, cfg.big, xb, a, cfg, s);
  }
}

}  // namespace nf4k
