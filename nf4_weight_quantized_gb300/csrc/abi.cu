// abi.cu -- the extern "C" boundary of libnf4: validation, device checks,
// configuration choice and asynchronous launches.  See include/nf4.h.
#include <cmath>
#include <cstdarg>
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"
#include "nf4.h"

namespace {

thread_local std::string g_last_error;
thread_local std::string g_describe;

nf4_status fail(nf4_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

// ---------------------------------------------------------------- codebook
//
// The 16 NormalFloat levels (QLoRA construction, Dettmers et al. 2023, sec. 3):
// N(0,1) quantiles at 8 evenly spaced probabilities from 1-d towards 1/2 and
// 7 from d towards 1/2, d = (1/32 + 1/30) / 2, plus an exact 0, divided by the
// largest and sorted.  The inverse normal CDF is found here by Newton's method
// on Phi(z) = erfc(-z / sqrt 2) / 2 started at 0 (Phi is concave above 0 and
// convex below, so the iterates approach the root from one side), in float64,
// and each level is rounded once to fp32.

double normal_cdf(double z) { return 0.5 * std::erfc(-z / std::sqrt(2.0)); }
double normal_pdf(double z) { return std::exp(-0.5 * z * z) / std::sqrt(2.0 * 3.14159265358979323846); }

double normal_quantile(double p) {
  double z = 0.0;
  for (int it = 0; it < 100; ++it) {
    const double dz = (normal_cdf(z) - p) / normal_pdf(z);
    z -= dz;
    if (std::fabs(dz) < 1e-16 * (1.0 + std::fabs(z))) break;
  }
  return z;
}

nf4k::Codebook make_codebook() {
  const double d = 0.5 * (1.0 / 32.0 + 1.0 / 30.0);
  double v[16];
  int n = 0;
  for (int j = 0; j < 8; ++j) v[n++] = normal_quantile(1.0 - d - j * (0.5 - d) / 8.0);
  for (int j = 0; j < 7; ++j) v[n++] = normal_quantile(d + j * (0.5 - d) / 7.0);
  v[n++] = 0.0;
  const double top = normal_quantile(1.0 - d);
  for (double& e : v) e /= top;
  for (int i = 1; i < 16; ++i)
    for (int j = i; j > 0 && v[j - 1] > v[j]; --j) std::swap(v[j - 1], v[j]);
  nf4k::Codebook cb;
  for (int i = 0; i < 16; ++i) cb.v[i] = (float)v[i];
  return cb;
}

const nf4k::Codebook& codebook() {
  static const nf4k::Codebook cb = make_codebook();
  return cb;
}

// ------------------------------------------------- device error registry

std::mutex& readers_mu() {
  static std::mutex mu;
  return mu;
}
std::vector<nf4k::DeviceErrorReader>& readers() {
  static std::vector<nf4k::DeviceErrorReader> v;
  return v;
}

// ------------------------------------------------------------------ device

struct DeviceInfo {
  int checked = 0;
  int cc_major = 0, cc_minor = 0, sms = 0;
};
std::mutex g_dev_mu;
DeviceInfo g_dev[64];

nf4_status current_device(int* dev) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return fail(NF4_ECUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (*dev < 0 || *dev >= 64) return fail(NF4_ECUDA, "device ordinal %d out of range", *dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_dev[*dev];
  if (!d.checked) {
    cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, *dev);
    cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, *dev);
    cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, *dev);
    e = cudaGetLastError();
    if (e != cudaSuccess) return fail(NF4_ECUDA, "device query: %s", cudaGetErrorString(e));
    d.checked = 1;
  }
  if (!(d.cc_major == 10 && d.cc_minor == 3))
    return fail(NF4_EARCH, "device %d is sm_%d%d; libnf4 is built for sm_103a only", *dev, d.cc_major,
                d.cc_minor);
  return NF4_OK;
}

// -------------------------------------------------------------- validation

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

nf4_status check_shape(int64_t M, int64_t K, const char* what) {
  if (M < 1 || M >= (int64_t(1) << 31))
    return fail(NF4_EINVAL, "%s: M = %lld must be in [1, 2^31)", what, (long long)M);
  if (K < 64 || K % 64 != 0 || K > NF4_MAX_K)
    return fail(NF4_EINVAL, "%s: K = %lld must be a positive multiple of 64 and <= %d", what, (long long)K,
                NF4_MAX_K);
  return NF4_OK;
}

nf4_status check_weight(const nf4_weight* W, const char* what) {
  if (!W) return fail(NF4_ENULL, "%s: weight descriptor is NULL", what);
  nf4_status st = check_shape(W->M, W->K, what);
  if (st) return st;
  if (!W->codes || !W->scales) return fail(NF4_ENULL, "%s: codes or scales is NULL", what);
  if (!aligned(W->codes, 16)) return fail(NF4_EALIGN, "%s: codes must be 16-byte aligned", what);
  if (!aligned(W->scales, 4)) return fail(NF4_EALIGN, "%s: scales must be 4-byte aligned", what);
  return NF4_OK;
}

nf4_status check_x(const void* x, nf4_dtype xt, const char* what) {
  if (!x) return fail(NF4_ENULL, "%s: x is NULL", what);
  if (xt != NF4_F32 && xt != NF4_BF16) return fail(NF4_EINVAL, "%s: unknown activation dtype %d", what, (int)xt);
  if (!aligned(x, 16)) return fail(NF4_EALIGN, "%s: x must be 16-byte aligned", what);
  return NF4_OK;
}

nf4_status check_out(const void* p, size_t align, const char* name, const char* what) {
  if (!p) return fail(NF4_ENULL, "%s: %s is NULL", what, name);
  if (!aligned(p, align)) return fail(NF4_EALIGN, "%s: %s must be %zu-byte aligned", what, name, align);
  return NF4_OK;
}

nf4_status launched(cudaError_t e, const char* what) {
  const std::string note = nf4k::take_launch_note();
  if (e != cudaSuccess) return fail(NF4_ECUDA, "%s: launch failed: %s%s", what, cudaGetErrorString(e), note.c_str());
  return NF4_OK;
}

// NF4_GEMV_KERNEL=register forces the register-prefetch kernel (tuning runs).
bool use_register_kernel() {
  static const bool v = [] {
    const char* e = std::getenv("NF4_GEMV_KERNEL");
    return e && std::strcmp(e, "register") == 0;
  }();
  return v;
}

// The three matrices of a fused q/k/v call with their biases and outputs.
struct QkvParts {
  const nf4_weight* W[3];
  const float* bias[3];
  float* out[3];
};

nf4_status run_gemv(int epi, const nf4_weight* W, const nf4_weight* W2, const void* x, nf4_dtype xt,
                    const float* resid, float* y, uint16_t* out, int64_t* index, void* ws, nf4_stream stream,
                    const char* what, const QkvParts* qkv = nullptr) {
  int dev = 0;
  nf4_status st = current_device(&dev);
  if (st) return st;
  nf4k::GemvArgs a{};
  a.codes = W->codes;
  a.scales = W->scales;
  if (W2) {
    a.codes2 = W2->codes;
    a.scales2 = W2->scales;
  }
  a.x = x;
  a.resid = resid;
  a.y = y;
  a.out_bf16 = out;
  a.index = index;
  a.ws = reinterpret_cast<unsigned long long*>(ws);
  a.M = (int)W->M;
  a.K = (int)W->K;
  a.cb = codebook();
  a.wait_polls = nf4k::data_wait_polls();
  bool scales16_extra = true;
  if (qkv) {  // one row space: q's rows, then k's, then v's
    int64_t end = 0;
    for (int i = 0; i < 3; ++i) {
      a.seg_codes[i] = qkv->W[i]->codes;
      a.seg_scales[i] = qkv->W[i]->scales;
      a.seg_bias[i] = qkv->bias[i];
      a.seg_out[i] = qkv->out[i];
      end += qkv->W[i]->M;
      a.seg_end[i] = (int)end;
      scales16_extra = scales16_extra && aligned(qkv->W[i]->scales, 16);
    }
    a.M = (int)end;
  }
  if (!use_register_kernel()) {
    const nf4k::ClusterConfig cc = nf4k::choose_cluster_config(epi, a.M, W->K, dev);
    if (cc.ok) {
      const cudaError_t e = nf4k::launch_gemv_cluster(epi, xt == NF4_BF16, a, cc, reinterpret_cast<cudaStream_t>(stream));
      if (e != cudaSuccess)
        return fail(NF4_ECUDA, "%s: launch failed (cluster kernel, %d clusters of %d blocks x %d threads): %s%s", what,
                    cc.clusters, cc.CL, cc.threads, cudaGetErrorString(e), nf4k::take_launch_note().c_str());
      return NF4_OK;
    }
  }
  const bool scales16 = aligned(W->scales, 16) && (!W2 || aligned(W2->scales, 16)) && scales16_extra;
  if (scales16 && !use_register_kernel()) {
    const nf4k::TmaConfig tc = nf4k::choose_tma_config(epi, xt == NF4_BF16, a.M, W->K, dev);
    if (tc.ok) {
      a.G = tc.G;
      a.gpc = tc.gpc;
      const cudaError_t e = nf4k::launch_gemv_tma(epi, xt == NF4_BF16, a, tc, reinterpret_cast<cudaStream_t>(stream));
      if (e != cudaSuccess)
        return fail(NF4_ECUDA, "%s: launch failed (bulk-copy kernel, %d blocks x %d threads, %d B shared): %s%s",
                    what, tc.blocks, tc.threads, tc.smem, cudaGetErrorString(e), nf4k::take_launch_note().c_str());
      return NF4_OK;
    }
  }
  const nf4k::GemvConfig cfg = nf4k::choose_gemv_config(epi, a.M, W->K, dev);
  a.G = cfg.G;
  a.gpc = cfg.gpc;
  const cudaError_t e = nf4k::launch_gemv(epi, xt == NF4_BF16, a, cfg, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess)
    return fail(NF4_ECUDA,
                "%s: launch failed (register kernel nch=%d rb=%d%s, %d blocks x %d threads, %d B shared): %s%s", what,
                cfg.nch, cfg.rb, cfg.big ? " capped" : "", cfg.blocks, cfg.G * cfg.gpc, cfg.smem,
                cudaGetErrorString(e), nf4k::take_launch_note().c_str());
  return NF4_OK;
}

}  // namespace

namespace nf4k {
void set_last_error(const char* msg) { g_last_error = msg; }

cudaError_t ensure_smem_limit(const void* fn, int bytes) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> done;  // (function, device) -> bytes set
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lk(mu);
  int& have = done[std::make_pair(fn, dev)];
  if (have >= bytes) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) have = bytes;
  return e;
}

bool pdl_enabled() {
  static const bool on = [] {
    const char* e = std::getenv("NF4_PDL");
    return !(e && *e == '0');
  }();
  return on;
}

namespace {
std::atomic<uint32_t> g_data_wait_polls{0};  // 0: kWaitPolls
}

uint32_t data_wait_polls() {
  const uint32_t v = g_data_wait_polls.load(std::memory_order_relaxed);
  return v ? v : kWaitPolls;
}

thread_local std::string g_launch_note;

void note_launch_failure(const void* fn, int threads, int smem, cudaError_t set_err, cudaError_t launch_err,
                         cudaError_t retry_err) {
  cudaFuncAttributes at{};
  const cudaError_t ae = cudaFuncGetAttributes(&at, fn);
  cudaGetLastError();
  char buf[512];
  std::snprintf(buf, sizeof buf,
                " [first attempt: limit %s, launch %s; retry %s; requested %d threads, %d B dynamic shared; "
                "function: %s, %d regs, %zu B static shared, max %d B dynamic, max %d threads]",
                cudaGetErrorName(set_err), cudaGetErrorName(launch_err), cudaGetErrorName(retry_err), threads, smem,
                cudaGetErrorName(ae), at.numRegs, at.sharedSizeBytes, at.maxDynamicSharedSizeBytes,
                at.maxThreadsPerBlock);
  g_launch_note = buf;
}

void note_stale_error(const void* fn, cudaError_t stale) {
  static const bool on = [] {
    const char* e = std::getenv("NF4_DEBUG_LAUNCH");
    return e && *e == '1';
  }();
  if (on) std::fprintf(stderr, "nf4: stale CUDA error before launching %p: %s\n", fn, cudaGetErrorName(stale));
}

std::string take_launch_note() {
  std::string s;
  s.swap(g_launch_note);
  return s;
}

void register_device_error_reader(DeviceErrorReader f) {
  std::lock_guard<std::mutex> lk(readers_mu());
  readers().push_back(f);
}
}  // namespace nf4k

extern "C" {

nf4_status nf4_check_device_errors(void) {
  int dev = 0;
  nf4_status st = current_device(&dev);
  if (st) return st;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return fail(NF4_ECUDA, "nf4_check_device_errors: %s", cudaGetErrorString(e));
  unsigned int bits = 0;
  {
    std::lock_guard<std::mutex> lk(readers_mu());
    for (auto f : readers()) bits |= f();
  }
  if (bits & nf4k::kErrWaitTimeout)
    return fail(NF4_ETIMEOUT, "a kernel gave up waiting on a shared-memory barrier; its outputs are invalid");
  if (bits & nf4k::kErrBadIndex)
    return fail(NF4_ERANGE, "nf4_dequant_rows was given a token id outside its table; those rows were written as zeros");
  return NF4_OK;
}

void nf4_debug_set_wait_limit(uint32_t polls) { nf4k::g_data_wait_polls.store(polls, std::memory_order_relaxed); }

nf4_status nf4_dequant_rows(const nf4_weight* E, const int64_t* ids, int64_t n, void* out, nf4_dtype ot,
                            nf4_stream stream) {
  const char* what = "nf4_dequant_rows";
  nf4_status st;
  if ((st = check_weight(E, what))) return st;
  if (n < 0) return fail(NF4_EINVAL, "%s: n = %lld is negative", what, (long long)n);
  if (ot != NF4_F32 && ot != NF4_BF16) return fail(NF4_EINVAL, "%s: output dtype %d is not NF4_F32 or NF4_BF16", what, (int)ot);
  if (n == 0) return NF4_OK;
  if ((st = check_out(ids, 8, "ids", what)) || (st = check_out(out, 16, "out", what))) return st;
  int dev = 0;
  if ((st = current_device(&dev))) return st;
  return launched(nf4k::launch_embed_rows(E->codes, E->scales, E->M, E->K, ids, n, out, ot == NF4_BF16, codebook(),
                                          reinterpret_cast<cudaStream_t>(stream)),
                  what);
}

nf4_status nf4_rmsnorm(const float* x, const uint16_t* w, int64_t rows, int64_t K, float eps, void* y,
                       nf4_dtype yt, nf4_stream stream) {
  const char* what = "nf4_rmsnorm";
  nf4_status st;
  if (rows < 1 || rows >= (int64_t(1) << 31))
    return fail(NF4_EINVAL, "%s: rows = %lld must be in [1, 2^31)", what, (long long)rows);
  if (K < 1 || K > NF4_MAX_K) return fail(NF4_EINVAL, "%s: K = %lld must be in [1, %d]", what, (long long)K, NF4_MAX_K);
  if (!(eps >= 0.0f) || !std::isfinite(eps)) return fail(NF4_EINVAL, "%s: eps must be finite and >= 0", what);
  if (yt != NF4_F32 && yt != NF4_BF16) return fail(NF4_EINVAL, "%s: output dtype %d is not NF4_F32 or NF4_BF16", what, (int)yt);
  if ((st = check_out(x, 4, "x", what)) || (st = check_out(w, 2, "w", what)) ||
      (st = check_out(y, yt == NF4_F32 ? 4 : 2, "y", what)))
    return st;
  if (yt == NF4_BF16 && static_cast<const void*>(y) == static_cast<const void*>(x))
    return fail(NF4_EINVAL, "%s: a bf16 output cannot overwrite the fp32 input in place", what);
  int dev = 0;
  if ((st = current_device(&dev))) return st;
  return launched(nf4k::launch_rmsnorm(x, w, rows, K, eps, y, yt == NF4_BF16, reinterpret_cast<cudaStream_t>(stream)),
                  what);
}

nf4_status nf4_gemv(const nf4_weight* W, const void* x, nf4_dtype xt, float* y, nf4_stream stream) {
  const char* what = "nf4_gemv";
  nf4_status st;
  if ((st = check_weight(W, what)) || (st = check_x(x, xt, what)) || (st = check_out(y, 4, "y", what))) return st;
  return run_gemv(nf4k::EPI_PLAIN, W, nullptr, x, xt, nullptr, y, nullptr, nullptr, nullptr, stream, what);
}

nf4_status nf4_gemv_residual(const nf4_weight* W, const void* x, nf4_dtype xt, const float* residual, float* y,
                             nf4_stream stream) {
  const char* what = "nf4_gemv_residual";
  nf4_status st;
  if ((st = check_weight(W, what)) || (st = check_x(x, xt, what)) || (st = check_out(y, 4, "y", what)) ||
      (st = check_out(residual, 4, "residual", what)))
    return st;
  return run_gemv(nf4k::EPI_RESID, W, nullptr, x, xt, residual, y, nullptr, nullptr, nullptr, stream, what);
}

nf4_status nf4_gemv_swiglu(const nf4_weight* Wg, const nf4_weight* Wu, const void* x, nf4_dtype xt, uint16_t* out,
                           nf4_stream stream) {
  const char* what = "nf4_gemv_swiglu";
  nf4_status st;
  if ((st = check_weight(Wg, what)) || (st = check_weight(Wu, what)) || (st = check_x(x, xt, what)) ||
      (st = check_out(out, 2, "out", what)))
    return st;
  if (Wg->M != Wu->M || Wg->K != Wu->K)
    return fail(NF4_EINVAL, "%s: gate is %lldx%lld but up is %lldx%lld", what, (long long)Wg->M,
                (long long)Wg->K, (long long)Wu->M, (long long)Wu->K);
  return run_gemv(nf4k::EPI_SWIGLU, Wg, Wu, x, xt, nullptr, nullptr, out, nullptr, nullptr, stream, what);
}

nf4_status nf4_gemv_glu_interleaved(const nf4_weight* W, const void* x, nf4_dtype xt, uint16_t* out,
                                    nf4_stream stream) {
  const char* what = "nf4_gemv_glu_interleaved";
  nf4_status st;
  if ((st = check_weight(W, what)) || (st = check_x(x, xt, what)) || (st = check_out(out, 2, "out", what)))
    return st;
  if (W->M % 2 != 0)
    return fail(NF4_EINVAL, "%s: W has %lld rows; interleaved gate/up rows come in pairs", what, (long long)W->M);
  return run_gemv(nf4k::EPI_GLU, W, nullptr, x, xt, nullptr, nullptr, out, nullptr, nullptr, stream, what);
}

nf4_status nf4_gemv_argmax(const nf4_weight* W, const void* x, nf4_dtype xt, float* logits, int64_t* index,
                           void* workspace, nf4_stream stream) {
  const char* what = "nf4_gemv_argmax";
  nf4_status st;
  if ((st = check_weight(W, what)) || (st = check_x(x, xt, what)) || (st = check_out(logits, 4, "logits", what)) ||
      (st = check_out(index, 8, "index", what)) || (st = check_out(workspace, 8, "workspace", what)))
    return st;
  return run_gemv(nf4k::EPI_ARGMAX, W, nullptr, x, xt, nullptr, logits, nullptr, index, workspace, stream, what);
}

nf4_status nf4_gemv_qkv(const nf4_weight* Wq, const nf4_weight* Wk, const nf4_weight* Wv, const float* bq,
                        const float* bk, const float* bv, const void* x, nf4_dtype xt, float* q, float* k, float* v,
                        nf4_stream stream) {
  const char* what = "nf4_gemv_qkv";
  nf4_status st;
  if ((st = check_weight(Wq, what)) || (st = check_weight(Wk, what)) || (st = check_weight(Wv, what)) ||
      (st = check_x(x, xt, what)) || (st = check_out(q, 4, "q", what)) || (st = check_out(k, 4, "k", what)) ||
      (st = check_out(v, 4, "v", what)))
    return st;
  if (Wk->K != Wq->K || Wv->K != Wq->K)
    return fail(NF4_EINVAL, "%s: q, k and v must share K (got %lld, %lld, %lld)", what, (long long)Wq->K,
                (long long)Wk->K, (long long)Wv->K);
  if (Wq->M + Wk->M + Wv->M >= ((int64_t)1 << 31))
    return fail(NF4_EINVAL, "%s: q.M + k.M + v.M = %lld rows exceeds 2^31 - 1", what,
                (long long)(Wq->M + Wk->M + Wv->M));
  const float* bias[3] = {bq, bk, bv};
  const char* bname[3] = {"bq", "bk", "bv"};
  for (int i = 0; i < 3; ++i)
    if (bias[i] && !aligned(bias[i], 4)) return fail(NF4_EALIGN, "%s: %s must be 4-byte aligned", what, bname[i]);
  QkvParts parts{{Wq, Wk, Wv}, {bq, bk, bv}, {q, k, v}};
  return run_gemv(nf4k::EPI_QKV, Wq, nullptr, x, xt, nullptr, nullptr, nullptr, nullptr, nullptr, stream, what,
                  &parts);
}

nf4_status nf4_gemm_chunk(const nf4_weight* W, const uint16_t* X, int N, float* Y, void* workspace,
                          nf4_stream stream) {
  const char* what = "nf4_gemm_chunk";
  nf4_status st;
  if ((st = check_weight(W, what))) return st;
  if (N < 1 || N > NF4_MAX_CHUNK_N) return fail(NF4_EINVAL, "%s: N = %d must be in [1, %d]", what, N, NF4_MAX_CHUNK_N);
  if ((st = check_out(X, 16, "X", what)) || (st = check_out(Y, 4, "Y", what))) return st;
  const size_t need = nf4_workspace_bytes(W->M, W->K, N);
  if (need && (st = check_out(workspace, 16, "workspace", what))) return st;
  int dev = 0;
  if ((st = current_device(&dev))) return st;
  return launched(nf4k::launch_chunk(W->codes, W->scales, (int)W->M, (int)W->K, X, N, Y, workspace, codebook(),
                                     reinterpret_cast<cudaStream_t>(stream), dev),
                  what);
}

size_t nf4_workspace_bytes(int64_t M, int64_t K, int N) {
  if (M < 1 || K < 64 || K % 64 || N < 1 || N > NF4_MAX_CHUNK_N) return 0;
  // argmax (N = 1): 64-bit key + block ticket; chunk: split-K partials + tickets
  const size_t chunk = nf4k::chunk_workspace_bytes(M, K, N);
  return N == 1 ? (chunk > 16 ? chunk : 16) : chunk;
}

nf4_status nf4_quantize(const float* W, int64_t M, int64_t K, uint8_t* codes, float* scales, nf4_stream stream) {
  const char* what = "nf4_quantize";
  nf4_status st;
  if ((st = check_shape(M, K, what))) return st;
  if ((st = check_out(W, 16, "W", what)) || (st = check_out(codes, 16, "codes", what)) ||
      (st = check_out(scales, 4, "scales", what)))
    return st;
  int dev = 0;
  if ((st = current_device(&dev))) return st;
  return launched(nf4k::launch_quantize(W, M, K, codes, scales, codebook(), reinterpret_cast<cudaStream_t>(stream), dev),
                  what);
}

void nf4_codebook(float out[16]) {
  const nf4k::Codebook& cb = codebook();
  for (int i = 0; i < 16; ++i) out[i] = cb.v[i];
}

const char* nf4_last_error(void) { return g_last_error.c_str(); }

const char* nf4_describe_config(int64_t M, int64_t K, int N) {
  return nf4_describe_launch(N == 1 ? "gemv" : "chunk", M, K, N);
}

const char* nf4_describe_launch(const char* op, int64_t M, int64_t K, int N) {
  static const struct {
    const char* name;
    int epi;
  } kOps[] = {{"gemv", nf4k::EPI_PLAIN},   {"residual", nf4k::EPI_RESID}, {"swiglu", nf4k::EPI_SWIGLU},
              {"glu", nf4k::EPI_GLU},      {"qkv", nf4k::EPI_QKV},        {"argmax", nf4k::EPI_ARGMAX},
              {"chunk", -1}};
  int epi = -2;
  for (const auto& o : kOps)
    if (op && std::strcmp(op, o.name) == 0) epi = o.epi;
  if (epi == -2 || (epi == -1) != (N > 1 || (op && std::strcmp(op, "chunk") == 0))) {
    g_describe = std::string("invalid operation: ") + (op ? op : "(null)") + " at N = " + std::to_string(N);
    return g_describe.c_str();
  }
  if (check_shape(M, K, "nf4_describe_launch") || N < 1 || N > NF4_MAX_CHUNK_N) {
    g_describe = std::string("invalid shape: ") + g_last_error;
    return g_describe.c_str();
  }
  int dev = 0;
  if (current_device(&dev)) {
    g_describe = std::string("no usable device: ") + g_last_error;
    return g_describe.c_str();
  }
  char buf[512];
  const nf4k::ClusterConfig cc =
      (epi >= 0 && !use_register_kernel()) ? nf4k::choose_cluster_config(epi, M, K, dev) : nf4k::ClusterConfig{};
  if (cc.ok) {
    std::snprintf(buf, sizeof buf,
                  "gemv M=%lld K=%lld: cluster split-K kernel, %d clusters of %d blocks (K split %d ways, %d rows per "
                  "cluster), %d threads per block, partial sums added through distributed shared memory, %s",
                  (long long)M, (long long)K, cc.clusters, cc.CL, cc.CL, cc.RPC, cc.threads,
                  nf4k::pdl_enabled() ? "programmatic dependent launch" : "plain launch");
  } else if (epi >= 0) {
    const nf4k::TmaConfig t = use_register_kernel() ? nf4k::TmaConfig{} : nf4k::choose_tma_config(epi, true, M, K, dev);
    if (t.ok) {
      std::snprintf(buf, sizeof buf,
                    "gemv M=%lld K=%lld (16-byte aligned scales): bulk-copy kernel, %d thread(s) per row, %d row(s) "
                    "per group and stage, %d group(s) (%d per stage) + 1 producer warp per block (%d threads), %d stages of %d rows "
                    "(%d B, %d row(s) per full barrier), %d blocks, %d B shared memory, %s table, %s",
                    (long long)M, (long long)K, t.G, t.rb, t.gpc, t.GPS, t.threads, t.S, t.SR, t.stage_bytes, t.subr, t.blocks,
                    t.smem, t.lut == 1 ? "fp16-level mixed-precision loop for bf16 x" : "fp32 pair",
                    nf4k::pdl_enabled() ? "programmatic dependent launch" : "plain launch");
    } else {
      const nf4k::GemvConfig c = nf4k::choose_gemv_config(epi, M, K, dev);
      std::snprintf(buf, sizeof buf,
                    "gemv M=%lld K=%lld: register kernel, %d thread(s) per row (%d chunk(s) of 32 weights each), %d "
                    "row(s) per batch, %d row group(s) per block, %d blocks of %d threads, %d B shared memory%s",
                    (long long)M, (long long)K, c.G, c.nch, c.rb, c.gpc, c.blocks, c.G * c.gpc, c.smem,
                    c.big ? ", register-capped" : "");
    }
  } else {
    std::snprintf(buf, sizeof buf, "%s", nf4k::describe_chunk(M, K, N, dev).c_str());
  }
  g_describe = buf;
  return g_describe.c_str();
}

}  // extern "C"
