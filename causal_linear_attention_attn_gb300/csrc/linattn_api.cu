// C ABI of liblinattn.so: argument validation, dispatch and status codes.
// Every entry point validates before it touches the GPU; see linattn.h for
// the contract of each call.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <cmath>
#include <cstdio>
#include <mutex>
#include <vector>

#include "internal.h"
#include "linattn.h"
#include "per_device.h"

namespace la {

namespace {

std::atomic<unsigned long long> g_launches{0};

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool supported_dim(int d) { return d == 32 || d == 64 || d == 128; }
// Feature counts of the calls on given features: the head sizes, and m = 256 (m = 2d at d = 128)
// when the state (m x d_v fp32) fits the CUDA-core kernels' shared memory (d_v <= 128).
bool supported_features(int m, int dv) { return supported_dim(m) || (m == 256 && dv <= 128); }

thread_local cudaError_t t_last_error = cudaSuccess;

la_status from_cuda(cudaError_t e) {
  if (e != cudaSuccess) {
    t_last_error = e;
    cudaGetLastError();  // clear a non-sticky error so later calls start clean
  }
  switch (e) {
    case cudaSuccess: return LA_OK;
    case cudaErrorMemoryAllocation: return LA_ERR_OUT_OF_MEMORY;
    case cudaErrorNoDevice:
    case cudaErrorInsufficientDriver: return LA_ERR_NO_DEVICE;
    default: return LA_ERR_LAUNCH;
  }
}

// Shared checks.  features: q and k are given features of any supported feature count.
la_status validate(const void *q, const void *k, const void *v, const float *out, const float *S,
                   const float *z, int B, int H, long N, int dk, int dv, float eps, la_dtype dt,
                   bool features = false) {
  if (B < 0 || H < 0 || N < 0 || dk <= 0 || dv <= 0) return LA_ERR_INVALID_VALUE;
  if (!std::isfinite(eps) || eps < 0.f) return LA_ERR_INVALID_VALUE;
  if (dt != LA_F32 && dt != LA_BF16) return LA_ERR_UNSUPPORTED;
  if (!(features ? supported_features(dk, dv) : supported_dim(dk)) || !supported_dim(dv)) return LA_ERR_UNSUPPORTED;
  const long BH = (long)B * H;
  if (BH > 0x7fffffffL) return LA_ERR_INVALID_VALUE;
  if (BH > 0 && (!S || !z)) return LA_ERR_INVALID_VALUE;
  if (BH > 0 && N > 0 && (!q || !k || !v || !out)) return LA_ERR_INVALID_VALUE;
  const void *ptrs[6] = {q, k, v, out, S, z};
  for (const void *p : ptrs)
    if (p && !aligned16(p)) return LA_ERR_MISALIGNED;
  return LA_OK;
}

la_status current_device(int *dev) {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) {
    t_last_error = cudaGetLastError();
    return LA_ERR_NO_DEVICE;
  }
  *dev = d;
  return LA_OK;
}

}  // namespace

void count_launch(unsigned n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

// --- device-time diagnostics --------------------------------------------------------
namespace {
struct PendingTiming {
  int kernel;
  cudaEvent_t start, end;
};
std::atomic<bool> g_profiling{false};
std::mutex g_prof_mu;
std::vector<PendingTiming> g_pending;
double g_prof_ms[kKNumKernels];
long long g_prof_n[kKNumKernels];

// Fold finished event pairs into the totals (caller holds g_prof_mu).
cudaError_t resolve_pending() {
  cudaError_t first = cudaSuccess;
  for (const PendingTiming &t : g_pending) {
    float ms = 0.f;
    cudaError_t e = cudaEventSynchronize(t.end);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, t.start, t.end);
    if (e == cudaSuccess) {
      g_prof_ms[t.kernel] += ms;
      g_prof_n[t.kernel] += 1;
    } else if (first == cudaSuccess) {
      first = e;
    }
    cudaEventDestroy(t.start);
    cudaEventDestroy(t.end);
  }
  g_pending.clear();
  return first;
}
}  // namespace

LaunchTimer::LaunchTimer(int kernel, cudaStream_t stream) : kernel_(kernel), stream_(stream) {
  if (!g_profiling.load(std::memory_order_relaxed)) return;
  if (cudaEventCreate(&start_) != cudaSuccess || cudaEventRecord(start_, stream_) != cudaSuccess) {
    if (start_) cudaEventDestroy(start_);
    start_ = nullptr;
    cudaGetLastError();
  }
}

void LaunchTimer::done(cudaError_t launch_error) {
  if (!start_) return;
  cudaEvent_t end = nullptr;
  if (launch_error != cudaSuccess || cudaEventCreate(&end) != cudaSuccess ||
      cudaEventRecord(end, stream_) != cudaSuccess) {
    cudaEventDestroy(start_);
    if (end) cudaEventDestroy(end);
    start_ = nullptr;
    return;
  }
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_pending.push_back({kernel_, start_, end});
  start_ = nullptr;
}

cudaError_t ensure_smem_optin(const void *kernel, int bytes) {
  static PerDeviceCache<std::pair<const void *, int>, cudaError_t> cache;
  int dev = 0;
  const cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  return cache.get(dev, std::make_pair(kernel, bytes), [&] {
    const cudaError_t r = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (r != cudaSuccess) cudaGetLastError();
    return r;
  });
}

DeviceInfo device_info(int dev) {
  static PerDeviceCache<int, DeviceInfo> cache;
  if (dev < 0 && cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return DeviceInfo{};
  }
  return cache.get(dev, 0, [dev] {
    DeviceInfo i;
    cudaDeviceGetAttribute(&i.sm_count, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&i.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&i.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&i.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cudaGetLastError();
    return i;
  });
}

}  // namespace la

using la::Problem;

extern "C" {

int la_version(void) { return (1 << 16) | 0; }

const char *la_last_error_detail(void) {
  static thread_local char buf[256];
  snprintf(buf, sizeof buf, "%s: %s", cudaGetErrorName(la::t_last_error), cudaGetErrorString(la::t_last_error));
  return buf;
}

la_status la_device_status(void *stream) {
  int dev;
  la_status st = la::current_device(&dev);
  if (st != LA_OK) return st;
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return la::from_cuda(e);
  unsigned int v = 0, vg = 0;
  unsigned int vf = 0;
  e = la::read_and_clear_device_status(&v);
  if (e == cudaSuccess) e = la::read_and_clear_global_tc_status(&vg);
  unsigned int vb = 0;
  if (e == cudaSuccess) e = la::read_and_clear_favor_status(&vf);
  if (e == cudaSuccess) e = la::read_and_clear_backward_status(&vb);
  if (e != cudaSuccess) return la::from_cuda(e);
  v |= vg | vf | vb;
  if (v & 1u) return LA_ERR_TIMEOUT;
  return v ? LA_ERR_LAUNCH : LA_OK;  // other bits: a kernel refused to run (e.g. misaligned shared memory)
}

la_status la_diag_force_segments(int segments) {
  if (segments < 0 || segments > 4096) return LA_ERR_INVALID_VALUE;
  la::force_segments(segments);
  return LA_OK;
}

la_status la_test_inject_missing_load(int chunk, unsigned int wait_us) {
  if (chunk < 0 || wait_us < 1 || wait_us > 1000000) return LA_ERR_INVALID_VALUE;
  la::arm_missing_load(chunk, wait_us);
  return LA_OK;
}

unsigned long long la_kernel_launches(void) { return la::g_launches.load(std::memory_order_relaxed); }

const char *la_status_string(la_status s) {
  switch (s) {
    case LA_OK: return "success";
    case LA_ERR_INVALID_VALUE: return "invalid argument (NULL pointer, negative size or bad eps)";
    case LA_ERR_UNSUPPORTED: return "unsupported head dimension or dtype";
    case LA_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case LA_ERR_OUT_OF_MEMORY: return "out of device memory for scratch";
    case LA_ERR_LAUNCH: return "kernel launch failed";
    case LA_ERR_TIMEOUT: return "a bounded device-side wait timed out";
    case LA_ERR_NO_DEVICE: return "no usable CUDA device";
    case LA_ERR_TOO_LARGE: return "problem needs more scratch than the fixed buffer of la_causal_noalloc";
  }
  return "unknown status";
}

static la_status causal_impl(const void *q, const void *k, const void *v, float *out, float *S, float *z,
                             int B, int H, int N, int d_k, int d_v, float eps, la_dtype dt, void *stream,
                             bool from_state) {
  la_status st = la::validate(q, k, v, out, S, z, B, H, N, d_k, d_v, eps, dt);
  if (st != LA_OK) return st;
  if ((long)B * H == 0) return LA_OK;
  int dev;
  if ((st = la::current_device(&dev)) != LA_OK) return st;
  Problem p{q, k, v, out, S, z, B * H, (long)N, d_k, d_v, eps, dt, (cudaStream_t)stream};
  if (N == 0) {
    if (from_state) return LA_OK;
    cudaError_t e = cudaMemsetAsync(S, 0, sizeof(float) * (size_t)p.BH * d_k * d_v, p.stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(z, 0, sizeof(float) * (size_t)p.BH * d_k, p.stream);
    return la::from_cuda(e);
  }
  if (la::causal_tc_supported(p)) return la::from_cuda(la::launch_causal_tc(p, from_state));
  return la::from_cuda(la::launch_causal_simt(p, p.N, from_state, true));
}

la_status la_causal(const void *q, const void *k, const void *v, float *out, float *S, float *z, int B, int H,
                    int N, int d_k, int d_v, float eps, la_dtype dt, void *stream) {
  return causal_impl(q, k, v, out, S, z, B, H, N, d_k, d_v, eps, dt, stream, false);
}

la_status la_causal_with_state(const void *q, const void *k, const void *v, float *out, float *S, float *z,
                               int B, int H, int N, int d_k, int d_v, float eps, la_dtype dt, void *stream) {
  return causal_impl(q, k, v, out, S, z, B, H, N, d_k, d_v, eps, dt, stream, true);
}

static la_status retention_impl(const void *q, const void *k, const void *v, float *out, float *S,
                                const float *gamma, int B, int H, int N, int d_k, int d_v, la_dtype dt,
                                void *stream, bool from_state) {
  if (B < 0 || H < 0 || N < 0 || d_k <= 0 || d_v <= 0) return LA_ERR_INVALID_VALUE;
  const long BH = (long)B * H;
  if (BH > 0x7fffffffL) return LA_ERR_INVALID_VALUE;
  if (BH == 0) return LA_OK;
  if (!S || !gamma || (N > 0 && (!q || !k || !v || !out))) return LA_ERR_INVALID_VALUE;
  for (int h = 0; h < H; ++h)
    if (!std::isfinite(gamma[h])) return LA_ERR_INVALID_VALUE;
  if (dt != LA_F32 && dt != LA_BF16) return LA_ERR_UNSUPPORTED;
  if (!la::supported_dim(d_k) || !la::supported_dim(d_v) || H > la::kMaxRetentionHeads) return LA_ERR_UNSUPPORTED;
  bool fast_decay = false;  // a head with gamma < 0.75 is outside the tensor-core path's weight range
  for (int h = 0; h < H; ++h) {
    if (!(gamma[h] >= 0.f && gamma[h] <= 1.f)) return LA_ERR_UNSUPPORTED;
    if (gamma[h] < 0.75f) fast_decay = true;
  }
  const void *ptrs[5] = {q, k, v, out, S};
  for (const void *ptr : ptrs)
    if (ptr && !la::aligned16(ptr)) return LA_ERR_MISALIGNED;
  int dev;
  la_status st = la::current_device(&dev);
  if (st != LA_OK) return st;
  Problem p{q, k, v, out, S, nullptr, (int)BH, (long)N, d_k, d_v, 0.f, dt, (cudaStream_t)stream};
  if (N == 0) {
    if (from_state) return LA_OK;
    return la::from_cuda(cudaMemsetAsync(S, 0, sizeof(float) * (size_t)BH * d_k * d_v, p.stream));
  }
  if (fast_decay || !la::causal_tc_supported(p))
    return la::from_cuda(la::launch_retention_simt(p, from_state, gamma, H));
  float log2g[la::kMaxRetentionHeads];
  for (int h = 0; h < H; ++h) log2g[h] = (float)std::log2((double)gamma[h]);
  return la::from_cuda(la::launch_retention_tc(p, from_state, log2g, H));
}

la_status la_retention(const void *q, const void *k, const void *v, float *out, float *S, const float *gamma,
                       int B, int H, int N, int d_k, int d_v, la_dtype dt, void *stream) {
  return retention_impl(q, k, v, out, S, gamma, B, H, N, d_k, d_v, dt, stream, false);
}

la_status la_retention_with_state(const void *q, const void *k, const void *v, float *out, float *S,
                                  const float *gamma, int B, int H, int N, int d_k, int d_v, la_dtype dt,
                                  void *stream) {
  return retention_impl(q, k, v, out, S, gamma, B, H, N, d_k, d_v, dt, stream, true);
}

la_status la_causal_features(const void *phi_q, const void *phi_k, const void *v, float *out, float *S, float *z,
                             int B, int H, int N, int m, int d_v, float eps, la_dtype dt, void *stream) {
  la_status st = la::validate(phi_q, phi_k, v, out, S, z, B, H, N, m, d_v, eps, dt, true);
  if (st != LA_OK) return st;
  if ((long)B * H == 0) return LA_OK;
  int dev;
  if ((st = la::current_device(&dev)) != LA_OK) return st;
  Problem p{phi_q, phi_k, v, out, S, z, B * H, (long)N, m, d_v, eps, dt, (cudaStream_t)stream};
  if (N == 0) {
    cudaError_t e = cudaMemsetAsync(S, 0, sizeof(float) * (size_t)p.BH * m * d_v, p.stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(z, 0, sizeof(float) * (size_t)p.BH * m, p.stream);
    return la::from_cuda(e);
  }
  if (la::causal_tc_supported(p)) return la::from_cuda(la::launch_causal_features_tc(p, false));
  return la::from_cuda(la::launch_causal_simt(p, p.N, false, true, true));
}

la_status la_global_features(const void *phi_q, const void *phi_k, const void *v, float *out, float *S, float *z,
                             int B, int H, int N, int m, int d_v, float eps, la_dtype dt, void *stream) {
  la_status st = la::validate(phi_q, phi_k, v, out, S, z, B, H, N, m, d_v, eps, dt, true);
  if (st != LA_OK) return st;
  if ((long)B * H == 0) return LA_OK;
  int dev;
  if ((st = la::current_device(&dev)) != LA_OK) return st;
  Problem p{phi_q, phi_k, v, out, S, z, B * H, (long)N, m, d_v, eps, dt, (cudaStream_t)stream};
  return la::from_cuda(la::launch_global_simt(p, true));
}

la_status la_favor_features(const void *x, const void *W, void *phi, int B, int H, int N, int d, int m,
                            la_dtype dt, void *stream) {
  if (B < 0 || H < 0 || N < 0 || d <= 0 || m <= 0) return LA_ERR_INVALID_VALUE;
  const long rows = (long)B * H * N;
  if ((long)B * H > 0x7fffffffL || rows > 0x7fffffffL) return LA_ERR_INVALID_VALUE;
  if (rows == 0) return LA_OK;
  if (!x || !W || !phi) return LA_ERR_INVALID_VALUE;
  if (dt != LA_F32 && dt != LA_BF16) return LA_ERR_UNSUPPORTED;
  if (!la::supported_dim(d) || !(la::supported_dim(m) || m == 256)) return LA_ERR_UNSUPPORTED;
  if (!la::aligned16(x) || !la::aligned16(W) || !la::aligned16(phi)) return LA_ERR_MISALIGNED;
  int dev;
  la_status st = la::current_device(&dev);
  if (st != LA_OK) return st;
  return la::from_cuda(la::launch_favor_features(x, W, phi, rows, d, m, dt, (cudaStream_t)stream));
}

la_status la_profile_enable(int on) {
  std::lock_guard<std::mutex> lk(la::g_prof_mu);
  if (on) {
    la::resolve_pending();
    for (int i = 0; i < la::kKNumKernels; ++i) la::g_prof_ms[i] = 0.0, la::g_prof_n[i] = 0;
  }
  la::g_profiling.store(on != 0);
  return LA_OK;
}

la_status la_profile_read(la_kernel kernel, double *ms_total, long long *launches) {
  if ((int)kernel < 0 || (int)kernel >= la::kKNumKernels || !ms_total || !launches) return LA_ERR_INVALID_VALUE;
  std::lock_guard<std::mutex> lk(la::g_prof_mu);
  const cudaError_t e = la::resolve_pending();
  *ms_total = la::g_prof_ms[kernel];
  *launches = la::g_prof_n[kernel];
  return la::from_cuda(e);
}

la_status la_causal_noalloc(const void *q, const void *k, const void *v, float *out, float *S, float *z, int B,
                            int H, int N, int d_k, int d_v, float eps, la_dtype dt, void *stream) {
  la_status st = la::validate(q, k, v, out, S, z, B, H, N, d_k, d_v, eps, dt);
  if (st != LA_OK) return st;
  if ((long)B * H == 0) return LA_OK;
  int dev;
  if ((st = la::current_device(&dev)) != LA_OK) return st;
  Problem p{q, k, v, out, S, z, B * H, (long)N, d_k, d_v, eps, dt, (cudaStream_t)stream};
  if (N == 0) {
    cudaError_t e = cudaMemsetAsync(S, 0, sizeof(float) * (size_t)p.BH * d_k * d_v, p.stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(z, 0, sizeof(float) * (size_t)p.BH * d_k, p.stream);
    return la::from_cuda(e);
  }
  if (!la::causal_tc_supported(p)) return la::from_cuda(la::launch_causal_simt(p, p.N, false, true));
  bool too_large = false;
  const cudaError_t e = la::launch_causal_tc_noalloc(p, dev, &too_large);
  if (too_large) return LA_ERR_TOO_LARGE;
  return la::from_cuda(e);
}

la_status la_global(const void *q, const void *k, const void *v, float *out, float *S, float *z, int B, int H,
                    int N, int d_k, int d_v, float eps, la_dtype dt, void *stream) {
  la_status st = la::validate(q, k, v, out, S, z, B, H, N, d_k, d_v, eps, dt);
  if (st != LA_OK) return st;
  if ((long)B * H == 0) return LA_OK;
  int dev;
  if ((st = la::current_device(&dev)) != LA_OK) return st;
  Problem p{q, k, v, out, S, z, B * H, (long)N, d_k, d_v, eps, dt, (cudaStream_t)stream};
  if (la::global_tc_supported(p)) return la::from_cuda(la::launch_global_tc(p));
  return la::from_cuda(la::launch_global_simt(p));
}

la_status la_decode_step(const void *q, const void *k, const void *v, float *out, float *S, float *z, int B,
                         int H, int d_k, int d_v, float eps, la_dtype dt, void *stream) {
  la_status st = la::validate(q, k, v, out, S, z, B, H, 1, d_k, d_v, eps, dt);
  if (st != LA_OK) return st;
  if ((long)B * H == 0) return LA_OK;
  int dev;
  if ((st = la::current_device(&dev)) != LA_OK) return st;
  Problem p{q, k, v, out, S, z, B * H, 1L, d_k, d_v, eps, dt, (cudaStream_t)stream};
  return la::from_cuda(la::launch_decode(p));
}

la_status la_causal_backward(const void *q, const void *k, const void *v, const float *dout, const float *S0,
                             const float *z0, const float *dS, const float *dz, float *dq, float *dk, float *dv,
                             float *dS0, float *dz0, int B, int H, int N, int d_k, int d_v, float eps, la_dtype dt,
                             void *stream) {
  if (B < 0 || H < 0 || N < 0 || d_k <= 0 || d_v <= 0) return LA_ERR_INVALID_VALUE;
  if (!std::isfinite(eps) || eps < 0.f) return LA_ERR_INVALID_VALUE;
  const long BH = (long)B * H;
  if (BH > 0x7fffffffL) return LA_ERR_INVALID_VALUE;
  if (BH == 0) return LA_OK;
  if (N > 0 && (!q || !k || !v || !dout || !dq || !dk || !dv)) return LA_ERR_INVALID_VALUE;
  if (dt != LA_F32 && dt != LA_BF16) return LA_ERR_UNSUPPORTED;
  if (!la::supported_dim(d_k) || !la::supported_dim(d_v)) return LA_ERR_UNSUPPORTED;
  const void *ptrs[13] = {q, k, v, dout, S0, z0, dS, dz, dq, dk, dv, dS0, dz0};
  for (const void *ptr : ptrs)
    if (ptr && !la::aligned16(ptr)) return LA_ERR_MISALIGNED;
  int dev;
  la_status st = la::current_device(&dev);
  if (st != LA_OK) return st;
  la::BackwardProblem b{{q, k, v, nullptr, nullptr, nullptr, (int)BH, (long)N, d_k, d_v, eps, dt, (cudaStream_t)stream},
                        dout, S0, z0, dS, dz, dq, dk, dv, dS0, dz0};
  if (la::backward_tc_supported(b)) return la::from_cuda(la::launch_causal_backward_tc(b));
  return la::from_cuda(la::launch_causal_backward(b));
}

la_status la_retention_decode_step(const void *q, const void *k, const void *v, float *out, float *S,
                                   const float *gamma, int B, int H, int d_k, int d_v, la_dtype dt, void *stream) {
  if (B < 0 || H < 0 || d_k <= 0 || d_v <= 0) return LA_ERR_INVALID_VALUE;
  const long BH = (long)B * H;
  if (BH > 0x7fffffffL) return LA_ERR_INVALID_VALUE;
  if (BH == 0) return LA_OK;
  if (!q || !k || !v || !out || !S || !gamma) return LA_ERR_INVALID_VALUE;
  for (int h = 0; h < H; ++h)
    if (!std::isfinite(gamma[h])) return LA_ERR_INVALID_VALUE;
  if (dt != LA_F32 && dt != LA_BF16) return LA_ERR_UNSUPPORTED;
  if (!la::supported_dim(d_k) || !la::supported_dim(d_v) || H > la::kMaxRetentionHeads) return LA_ERR_UNSUPPORTED;
  for (int h = 0; h < H; ++h)
    if (!(gamma[h] >= 0.f && gamma[h] <= 1.f)) return LA_ERR_UNSUPPORTED;
  const void *ptrs[5] = {q, k, v, out, S};
  for (const void *ptr : ptrs)
    if (!la::aligned16(ptr)) return LA_ERR_MISALIGNED;
  int dev;
  la_status st = la::current_device(&dev);
  if (st != LA_OK) return st;
  Problem p{q, k, v, out, S, nullptr, (int)BH, 1L, d_k, d_v, 0.f, dt, (cudaStream_t)stream};
  return la::from_cuda(la::launch_retention_decode(p, gamma, H));
}

}  // extern "C"
