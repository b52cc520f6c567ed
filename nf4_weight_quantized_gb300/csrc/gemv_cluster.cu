// gemv_cluster.cu -- configuration and launch of the cluster split-K N=1 kernel
// (gemv_cluster.cuh) for projections with few rows.
#include <cstdlib>

#include "gemv_cluster.cuh"

namespace nf4k {

namespace {

int env_or(const char* name, int dflt) {
  const char* v = std::getenv(name);
  return (v && *v) ? std::atoi(v) : dflt;
}

template <int EPI>
const void* cluster_ptr(bool xb) {
  return xb ? reinterpret_cast<const void*>(&gemv_cluster_kernel<EPI, true>)
            : reinterpret_cast<const void*>(&gemv_cluster_kernel<EPI, false>);
}

const void* cluster_kernel_ptr(int epi, bool xb) {
  switch (epi) {
    case EPI_PLAIN: return cluster_ptr<EPI_PLAIN>(xb);
    case EPI_RESID: return cluster_ptr<EPI_RESID>(xb);
    case EPI_QKV: return cluster_ptr<EPI_QKV>(xb);
    default: return nullptr;
  }
}

}  // namespace

// Opt-in (NF4_CLUSTER=1): plain, residual and fused q/k/v projections of at
// most NF4_CLUSTER_MAX_WEIGHTS weights (default 8 Mi) with K <= 8192 (a
// block's K slice is at most 32 chunks).  Cluster size NF4_CLUSTER_SIZE
// (default 8, the portable maximum) or the largest power of two not above
// K / 32; one wave of SMs / CL clusters.  Measured graph-replayed on a GB300
// against the bulk-copy kernel, it is slower on every small shape tried
// (256 x 2048: 6.2 us with clusters of 8, 3.6 with clusters of 2, 3.0
// bulk-copy; 2048 x 2048: 7.7 / 4.4 / 3.7 us): a cluster needs all its SMs free
// at once, which defeats the early start of programmatic dependent launch,
// and adds two cluster barriers.  So it is not chosen by default.
ClusterConfig choose_cluster_config(int epi, int64_t M, int64_t K, int device) {
  ClusterConfig c{};
  c.ok = false;
  const int mode = env_or("NF4_CLUSTER", 0);
  if (mode != 1) return c;
  if (epi != EPI_PLAIN && epi != EPI_RESID && epi != EPI_QKV) return c;
  const int64_t H = K / 32;
  int CL = env_or("NF4_CLUSTER_SIZE", 8);
  while (CL > 1 && CL > H) CL >>= 1;
  if (CL < 1 || (H + CL - 1) / CL > 32) return c;
  const int64_t max_w = (int64_t)env_or("NF4_CLUSTER_MAX_WEIGHTS", 8 << 20);
  if (M * K > max_w) return c;
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
  sms = sms > 0 ? sms : 1;
  int64_t clusters = sms / CL;
  clusters = clusters < 1 ? 1 : clusters;
  int64_t rpc = (M + clusters - 1) / clusters;
  clusters = (M + rpc - 1) / rpc;
  // rows per pass, as the kernel derives it: TPR threads per row (the next
  // power of two above the largest K slice), 32 / TPR rows per warp
  const int64_t hr = (H + CL - 1) / CL;
  int tpr = 1;
  while (tpr < hr) tpr <<= 1;
  const int64_t rpp = (int64_t)(32 / tpr) * (kClusterThreads / 32);
  if (rpc > rpp * kClusterPasses) return c;  // more rows than one wave of clusters holds in registers
  c.CL = CL;
  c.RPC = (int)rpc;
  c.clusters = (int)clusters;
  c.threads = kClusterThreads;
  c.smem = (int)(rpc * 4);
  c.ok = true;
  return c;
}

cudaError_t launch_gemv_cluster(int epi, bool xb, const GemvArgs& a, const ClusterConfig& c, cudaStream_t s) {
  const void* fn = cluster_kernel_ptr(epi, xb);
  if (!fn) return cudaErrorInvalidValue;
  return checked_launch(fn, c.threads, c.smem, [&] {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)(c.clusters * c.CL));
    cfg.blockDim = dim3((unsigned)c.threads);
    cfg.dynamicSmemBytes = (size_t)c.smem;
    cfg.stream = s;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)c.CL;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = pdl_enabled() ? 2 : 1;
    const int CL = c.CL, RPC = c.RPC;
    switch (epi) {
      case EPI_PLAIN:
        if (xb) cudaLaunchKernelEx(&cfg, gemv_cluster_kernel<EPI_PLAIN, true>, a, CL, RPC);
        else cudaLaunchKernelEx(&cfg, gemv_cluster_kernel<EPI_PLAIN, false>, a, CL, RPC);
        break;
      case EPI_RESID:
        if (xb) cudaLaunchKernelEx(&cfg, gemv_cluster_kernel<EPI_RESID, true>, a, CL, RPC);
        else cudaLaunchKernelEx(&cfg, gemv_cluster_kernel<EPI_RESID, false>, a, CL, RPC);
        break;
      default:
        if (xb) cudaLaunchKernelEx(&cfg, gemv_cluster_kernel<EPI_QKV, true>, a, CL, RPC);
        else cudaLaunchKernelEx(&cfg, gemv_cluster_kernel<EPI_QKV, false>, a, CL, RPC);
        break;
    }
  });
}

}  // namespace nf4k
