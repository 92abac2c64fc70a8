// Global (non-causal) linear attention on CUDA cores, fp32 arithmetic.
//
// S = phi(K)^T V and z = phi(K)^T 1 over the whole sequence, then every
// position reads O = phi(Q) S / (phi(Q) z + eps) ("线性注意力从头到尾讲清楚"
// §5 and §8; "Linear Attention Math", "The associativity trick, written
// out").  The sum over N is split across CTAs that add their partial states
// into S, z with fp32 atomics (S, z are zeroed first on the same stream).
// Each build CTA accumulates the 128 state rows [128 z, 128 z + 128), z =
// blockIdx.z, so that a 256-row state (given features, m = 256) keeps 64
// entries a thread in registers.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace la {
namespace {

constexpr int kT = 64;
constexpr int kThreads = 256;
constexpr int kSliceRows = 128;                           // state rows a build CTA accumulates
constexpr int kMaxEntries = kSliceRows * 128 / kThreads;  // state entries per thread (d_v <= 128)

// Tokens per read CTA: 128, or 64 where the state is 256 rows (given features, m = 256).
__host__ __device__ inline int read_tokens(int dk) { return dk > 128 ? 64 : 128; }

template <typename Tin>
__global__ void __launch_bounds__(kThreads)
    global_state_kernel(const Tin *__restrict__ k, const Tin *__restrict__ v, float *__restrict__ S_g,
                        float *__restrict__ z_g, long N, int dk, int dv, int splits, int identity) {
  extern __shared__ float sm[];
  const int dkp = dk + 1;
  float *Ks = sm;             // [kT][dkp]
  float *Vs = Ks + kT * dkp;  // [kT][dv]
  const long bh = blockIdx.x;
  const int tid = threadIdx.x;
  const long tb = N * blockIdx.y / splits, te = N * (blockIdx.y + 1) / splits;
  const Tin *kh = k + bh * N * dk;
  const Tin *vh = v + bh * N * dv;
  const int i0 = blockIdx.z * kSliceRows, dks = min(kSliceRows, dk - i0);  // this CTA's state rows
  const int ne = dks * dv / kThreads;  // >= 4 for the supported sizes

  float acc[kMaxEntries];
#pragma unroll
  for (int r = 0; r < kMaxEntries; ++r) acc[r] = 0.f;
  float zacc = 0.f;

  for (long t0 = tb; t0 < te; t0 += kT) {
    const int T = (int)min((long)kT, te - t0);
    __syncthreads();
    for (int e = tid; e < T * dk; e += kThreads) {
      const int t = e / dk, i = e - t * dk;
      const float x = ldf(kh + (t0 + t) * dk + i);
      Ks[t * dkp + i] = identity ? x : phi(x);  // identity: k is a given feature
    }
    for (int e = tid; e < T * dv; e += kThreads) Vs[e] = ldf(vh + t0 * dv + e);
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kMaxEntries; ++r) {
      if (r < ne) {
        const int e = tid + r * kThreads;
        const int i = i0 + e / dv, c = e % dv;
        float s = acc[r];
        for (int j = 0; j < T; ++j) s = fmaf(Ks[j * dkp + i], Vs[j * dv + c], s);
        acc[r] = s;
      }
    }
    if (tid < dks)
      for (int j = 0; j < T; ++j) zacc += Ks[j * dkp + i0 + tid];
  }
  float *Sh = S_g + bh * (long)dk * dv + (long)i0 * dv;
#pragma unroll
  for (int r = 0; r < kMaxEntries; ++r)
    if (r < ne) atomicAdd(Sh + tid + r * kThreads, acc[r]);
  if (tid < dks) atomicAdd(z_g + bh * dk + i0 + tid, zacc);
}

template <typename Tin>
__global__ void __launch_bounds__(kThreads)
    global_read_kernel(const Tin *__restrict__ q, const float *__restrict__ S_g,
                       const float *__restrict__ z_g, float *__restrict__ out, long N, int dk, int dv,
                       float eps, int identity) {
  extern __shared__ float sm[];
  const int dkp = dk + 1, rt = read_tokens(dk);
  float *S = sm;                    // [dk][dv]
  float *z = S + dk * dv;           // [dk]
  float *Qs = z + dk;               // [rt][dkp]
  float *den = Qs + rt * dkp;       // [rt]
  const long bh = blockIdx.x;
  const int tid = threadIdx.x;
  const long t0 = (long)blockIdx.y * rt;
  const int T = (int)min((long)rt, N - t0);
  for (int e = tid; e < dk * dv; e += kThreads) S[e] = S_g[bh * dk * dv + e];
  for (int i = tid; i < dk; i += kThreads) z[i] = z_g[bh * dk + i];
  const Tin *qh = q + (bh * N + t0) * dk;
  for (int e = tid; e < T * dk; e += kThreads) {
    const int t = e / dk, i = e - t * dk;
    const float x = ldf(qh + e);
    Qs[t * dkp + i] = identity ? x : phi(x);
  }
  __syncthreads();
  for (int t = tid; t < T; t += kThreads) {
    float d = 0.f;
    for (int i = 0; i < dk; ++i) d = fmaf(Qs[t * dkp + i], z[i], d);
    den[t] = d + eps;
  }
  __syncthreads();
  float *oh = out + (bh * N + t0) * dv;
  for (int e = tid; e < T * dv; e += kThreads) {
    const int t = e / dv, c = e - t * dv;
    float n = 0.f;
    for (int i = 0; i < dk; ++i) n = fmaf(Qs[t * dkp + i], S[i * dv + c], n);
    oh[e] = n / den[t];
  }
}

template <typename Tin>
cudaError_t launch_t(const Problem &p, bool identity) {
  const DeviceInfo &di = device_info(-1);
  cudaError_t e = cudaMemsetAsync(p.S, 0, sizeof(float) * (size_t)p.BH * p.dk * p.dv, p.stream);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(p.z, 0, sizeof(float) * (size_t)p.BH * p.dk, p.stream);
  if (e != cudaSuccess) return e;
  if (p.N == 0) return cudaSuccess;
  // enough CTAs to cover the SMs a few times over, each with >= kT tokens
  long splits = (4L * di.sm_count + p.BH - 1) / p.BH;
  splits = std::max(1L, std::min(splits, (p.N + kT - 1) / kT));
  const size_t smem1 = sizeof(float) * ((size_t)kT * (p.dk + 1) + (size_t)kT * p.dv);
  e = cudaFuncSetAttribute(global_state_kernel<Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem1);
  if (e != cudaSuccess) return e;
  const unsigned slices = (unsigned)((p.dk + kSliceRows - 1) / kSliceRows);
  LaunchTimer t1(kKGlobalState, p.stream);
  global_state_kernel<Tin><<<dim3(p.BH, (unsigned)splits, slices), kThreads, smem1, p.stream>>>(
      (const Tin *)p.k, (const Tin *)p.v, p.S, p.z, p.N, p.dk, p.dv, (int)splits, identity ? 1 : 0);
  e = cudaGetLastError();
  t1.done(e);
  if (e != cudaSuccess) return e;
  count_launch();
  const int rt = read_tokens(p.dk);
  const size_t smem2 = sizeof(float) * ((size_t)p.dk * p.dv + p.dk + (size_t)rt * (p.dk + 1) + rt);
  e = cudaFuncSetAttribute(global_read_kernel<Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem2);
  if (e != cudaSuccess) return e;
  const unsigned tiles = (unsigned)((p.N + rt - 1) / rt);
  LaunchTimer t2(kKGlobalRead, p.stream);
  global_read_kernel<Tin><<<dim3(p.BH, tiles), kThreads, smem2, p.stream>>>((const Tin *)p.q, p.S, p.z, p.out,
                                                                          p.N, p.dk, p.dv, p.eps, identity ? 1 : 0);
  e = cudaGetLastError();
  t2.done(e);
  if (e == cudaSuccess) count_launch();
  return e;
}

}  // namespace

cudaError_t launch_global_simt(const Problem &p, bool identity) {
  if (p.dt == LA_F32) return launch_t<float>(p, identity);
  return launch_t<__nv_bfloat16>(p, identity);
}

}  // namespace la
