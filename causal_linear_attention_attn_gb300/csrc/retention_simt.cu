// Retention prefill on CUDA cores, exact fp32, for every case the tensor-core
// path does not take: fp32 inputs, head sizes other than 128, and decays
// below 0.75 (down to 0).
//
// Retention is the causal recurrence with a per-head decay gamma and no
// denominator, S_t = gamma S_{t-1} + k_t v_t^T, out_t = q_t^T S_t ("Linear
// Attention Math", "The kernel cousins: SSMs and RetNet"), with q and k used
// as given.  Over a chunk of T tokens (local rows t, j) that starts from the
// state S:
//   out_t = gamma^(t+1) q_t^T S + sum_{j <= t} gamma^(t-j) (q_t . k_j) v_j
//   S    <- gamma^T S + sum_j gamma^(T-1-j) k_j v_j^T.
// With 64-token chunks every power lies in [gamma^64, 1]: no power exceeds 1,
// so no decay, however small, leaves float range (the small ones underflow to
// zero, as the recurrence itself does).  One CTA per head, chunks in order.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace la {
namespace {

constexpr int kT = 64;  // tokens per chunk
constexpr int kThreads = 256;

struct RetParams {
  int H;                           // head h of every batch row decays by gamma[h]
  float gamma[kMaxRetentionHeads];
};

size_t ret_smem_bytes(int dk, int dv) {
  const size_t floats = (size_t)dk * dv + 2 * (size_t)kT * (dk + 1) + (size_t)kT * dv + (size_t)kT * (kT + 1) +
                        (kT + 1);
  return floats * sizeof(float);
}

template <typename Tin>
__global__ void __launch_bounds__(kThreads)
    retention_simt_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k, const Tin *__restrict__ v,
                          float *__restrict__ out, float *__restrict__ S_g, long N, int dk, int dv, int from_state,
                          const __grid_constant__ RetParams rp) {
  extern __shared__ float sm[];
  const int dkp = dk + 1;           // padded rows: conflict-free column walks
  float *S = sm;                    // [dk][dv] carried state
  float *Qs = S + dk * dv;          // [kT][dkp]
  float *Ks = Qs + kT * dkp;        // [kT][dkp]
  float *Vs = Ks + kT * dkp;        // [kT][dv]
  float *A = Vs + kT * dv;          // [kT][kT + 1] decayed scores gamma^(t-j) (q_t . k_j), j <= t
  float *pw = A + kT * (kT + 1);    // [kT + 1] gamma^n

  const long bh = blockIdx.x;
  const int tid = threadIdx.x;
  const float g = rp.gamma[bh % rp.H];
  const Tin *qh = q + bh * N * dk, *kh = k + bh * N * dk, *vh = v + bh * N * dv;
  float *oh = out + bh * N * dv;
  float *Sh = S_g + bh * (long)dk * dv;

  for (int e = tid; e < dk * dv; e += kThreads) S[e] = from_state ? Sh[e] : 0.f;
  for (int n = tid; n <= kT; n += kThreads) pw[n] = powf(g, (float)n);  // powf(0, 0) = 1

  for (long t0 = 0; t0 < N; t0 += kT) {
    const int T = (int)min((long)kT, N - t0);
    __syncthreads();  // the previous chunk is fully consumed (and pw is written)
    for (int e = tid; e < T * dk; e += kThreads) {
      const int t = e / dk, i = e - t * dk;
      Qs[t * dkp + i] = ldf(qh + (t0 + t) * dk + i);
      Ks[t * dkp + i] = ldf(kh + (t0 + t) * dk + i);
    }
    for (int e = tid; e < T * dv; e += kThreads) Vs[e] = ldf(vh + t0 * dv + e);
    __syncthreads();

    for (int e = tid; e < T * T; e += kThreads) {
      const int t = e / T, j = e - t * T;
      float a = 0.f;
      if (j <= t) {
        for (int i = 0; i < dk; ++i) a = fmaf(Qs[t * dkp + i], Ks[j * dkp + i], a);
        a *= pw[t - j];
      }
      A[t * (kT + 1) + j] = a;
    }
    __syncthreads();

    // out_t = gamma^(t+1) q_t^T S + sum_{j <= t} A[t][j] v_j
    for (int e = tid; e < T * dv; e += kThreads) {
      const int t = e / dv, c = e - t * dv;
      float n = 0.f;
      for (int i = 0; i < dk; ++i) n = fmaf(Qs[t * dkp + i], S[i * dv + c], n);
      float m = 0.f;
      for (int j = 0; j <= t; ++j) m = fmaf(A[t * (kT + 1) + j], Vs[j * dv + c], m);
      oh[(t0 + t) * dv + c] = fmaf(pw[t + 1], n, m);
    }
    __syncthreads();

    // S <- gamma^T S + sum_j gamma^(T-1-j) k_j v_j^T
    for (int e = tid; e < dk * dv; e += kThreads) {
      const int i = e / dv, c = e - i * dv;
      float s = 0.f;
      for (int j = 0; j < T; ++j) s = fmaf(Ks[j * dkp + i] * pw[T - 1 - j], Vs[j * dv + c], s);
      S[e] = fmaf(pw[T], S[e], s);
    }
  }
  __syncthreads();
  for (int e = tid; e < dk * dv; e += kThreads) Sh[e] = S[e];
}

template <typename Tin>
cudaError_t launch_t(const Problem &p, bool from_state, const float *gamma, int H) {
  const size_t smem = ret_smem_bytes(p.dk, p.dv);
  cudaError_t e = ensure_smem_optin((const void *)retention_simt_kernel<Tin>, (int)smem);
  if (e != cudaSuccess) return e;
  RetParams rp;
  rp.H = H;
  for (int h = 0; h < kMaxRetentionHeads; ++h) rp.gamma[h] = h < H ? gamma[h] : 0.f;
  LaunchTimer timer(kKRetentionMain, p.stream);
  retention_simt_kernel<Tin><<<p.BH, kThreads, smem, p.stream>>>(
      (const Tin *)p.q, (const Tin *)p.k, (const Tin *)p.v, p.out, p.S, p.N, p.dk, p.dv, from_state ? 1 : 0, rp);
  e = cudaGetLastError();
  timer.done(e);
  if (e == cudaSuccess) count_launch();
  return e;
}

}  // namespace

cudaError_t launch_retention_simt(const Problem &p, bool from_state, const float *gamma, int H) {
  if (!gamma || H < 1 || H > kMaxRetentionHeads) return cudaErrorInvalidValue;
  return p.dt == LA_F32 ? launch_t<float>(p, from_state, gamma, H) : launch_t<__nv_bfloat16>(p, from_state, gamma, H);
}

}  // namespace la
