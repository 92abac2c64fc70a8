// Exact fp32 chunked causal linear attention on CUDA cores.
//
// The causal recurrence ("线性注意力从头到尾讲清楚" §7; "Linear Attention
// Math", "The recurrent form") evaluated chunk by chunk: a chunk of T tokens
// reads the state carried from earlier chunks and adds its own masked
// (inclusive) pairwise part, then folds its keys and values into the state
// ("Linear Attention: From Pairwise Reads to a Recurrent State", "A
// recurrence need not force token-serial training").  One CTA per head, all
// arithmetic in fp32.  This is the path for float32 inputs, the exact pass
// over the first chunk of bf16 sequences, and the general fallback.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace la {
namespace {

constexpr int kT = 64;  // tokens per chunk
constexpr int kThreads = 256;

size_t simt_smem_bytes(int dk, int dv) {
  const size_t floats = (size_t)dk * dv + dk + 2 * (size_t)kT * (dk + 1) + (size_t)kT * dv +
                        (size_t)kT * (kT + 1) + kT;
  return floats * sizeof(float);
}

template <typename Tin>
__global__ void __launch_bounds__(kThreads)
    causal_simt_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k, const Tin *__restrict__ v,
                       float *__restrict__ out, float *__restrict__ S_g, float *__restrict__ z_g,
                       long N, long n_proc, int dk, int dv, float eps, int from_state,
                       int write_state) {
  extern __shared__ float sm[];
  const int dkp = dk + 1;  // padded row: conflict-free column walks
  float *S = sm;                  // [dk][dv]  carried state
  float *z = S + dk * dv;         // [dk]      carried normalizer
  float *Qs = z + dk;             // [kT][dkp] phi(q) of the chunk
  float *Ks = Qs + kT * dkp;      // [kT][dkp] phi(k)
  float *Vs = Ks + kT * dkp;      // [kT][dv]
  float *A = Vs + kT * dv;        // [kT][kT+1] masked pairwise weights
  float *den = A + kT * (kT + 1); // [kT]

  const long bh = blockIdx.x;
  const int tid = threadIdx.x;
  const Tin *qh = q + bh * N * dk;
  const Tin *kh = k + bh * N * dk;
  const Tin *vh = v + bh * N * dv;
  float *oh = out + bh * N * dv;
  float *Sh = S_g + bh * (long)dk * dv;
  float *zh = z_g + bh * (long)dk;

  for (int e = tid; e < dk * dv; e += kThreads) S[e] = from_state ? Sh[e] : 0.f;
  for (int i = tid; i < dk; i += kThreads) z[i] = from_state ? zh[i] : 0.f;

  for (long t0 = 0; t0 < n_proc; t0 += kT) {
    const int T = (int)min((long)kT, n_proc - t0);
    __syncthreads();  // the previous chunk is fully consumed
    for (int e = tid; e < T * dk; e += kThreads) {
      const int t = e / dk, i = e - t * dk;
      Qs[t * dkp + i] = phi(ldf(qh + (t0 + t) * dk + i));
      Ks[t * dkp + i] = phi(ldf(kh + (t0 + t) * dk + i));
    }
    for (int e = tid; e < T * dv; e += kThreads) Vs[e] = ldf(vh + t0 * dv + e);
    __syncthreads();

    // A[t][j] = phi(q_t) . phi(k_j) for j <= t (the read includes token t)
    for (int e = tid; e < T * T; e += kThreads) {
      const int t = e / T, j = e - t * T;
      float a = 0.f;
      if (j <= t)
        for (int i = 0; i < dk; ++i) a = fmaf(Qs[t * dkp + i], Ks[j * dkp + i], a);
      A[t * (kT + 1) + j] = a;
    }
    __syncthreads();

    // denominator: phi(q_t) . z_prev + sum_{j<=t} A[t][j] + eps
    for (int t = tid; t < T; t += kThreads) {
      float d = 0.f;
      for (int i = 0; i < dk; ++i) d = fmaf(Qs[t * dkp + i], z[i], d);
      float a = 0.f;
      for (int j = 0; j <= t; ++j) a += A[t * (kT + 1) + j];
      den[t] = (d + a) + eps;
    }
    __syncthreads();

    // numerator: phi(q_t)^T S_prev + sum_{j<=t} A[t][j] v_j
    for (int e = tid; e < T * dv; e += kThreads) {
      const int t = e / dv, c = e - t * dv;
      float n = 0.f;
      for (int i = 0; i < dk; ++i) n = fmaf(Qs[t * dkp + i], S[i * dv + c], n);
      float m = 0.f;
      for (int j = 0; j <= t; ++j) m = fmaf(A[t * (kT + 1) + j], Vs[j * dv + c], m);
      oh[(t0 + t) * dv + c] = (n + m) / den[t];
    }
    __syncthreads();

    // fold the chunk into the carried state
    for (int e = tid; e < dk * dv; e += kThreads) {
      const int i = e / dv, c = e - i * dv;
      float s = 0.f;
      for (int j = 0; j < T; ++j) s = fmaf(Ks[j * dkp + i], Vs[j * dv + c], s);
      S[e] += s;
    }
    for (int i = tid; i < dk; i += kThreads) {
      float s = 0.f;
      for (int j = 0; j < T; ++j) s += Ks[j * dkp + i];
      z[i] += s;
    }
  }
  __syncthreads();
  if (write_state) {
    for (int e = tid; e < dk * dv; e += kThreads) Sh[e] = S[e];
    for (int i = tid; i < dk; i += kThreads) zh[i] = z[i];
  }
}

template <typename Tin>
cudaError_t launch_t(const Problem &p, long n_proc, bool from_state, bool write_state) {
  const size_t smem = simt_smem_bytes(p.dk, p.dv);
  cudaError_t e = cudaFuncSetAttribute(causal_simt_kernel<Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  LaunchTimer timer(kKCausalSimt, p.stream);
  causal_simt_kernel<Tin><<<p.BH, kThreads, smem, p.stream>>>(
      (const Tin *)p.q, (const Tin *)p.k, (const Tin *)p.v, p.out, p.S, p.z, p.N, n_proc, p.dk, p.dv, p.eps,
      from_state ? 1 : 0, write_state ? 1 : 0);
  e = cudaGetLastError();
  timer.done(e);
  if (e == cudaSuccess) count_launch();
  return e;
}

// Exact fp32 outputs for tokens [0, ne) of a head (ne <= 64).  The leading
// tokens of a sequence read a state built from few tokens, so their outputs
// are O(1) while later ones average down; they get full fp32 weights here
// instead of the tensor cores' bf16 operands.  One warp per query row t:
// lanes split the keys j <= t for the weights phi(q_t).phi(k_j), then split
// the output columns for sum_j w_j v_j.  A CTA covers 16 rows of one head.
constexpr int kHeadRows = 16;

template <typename Tin>
__global__ void __launch_bounds__(kHeadRows * 32)
    causal_exact_head_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k, const Tin *__restrict__ v,
                             float *__restrict__ out, const float *__restrict__ S0, const float *__restrict__ z0,
                             long N, int ne, int dk, int dv, float eps) {
  extern __shared__ float sm[];
  const int dkp = dk + 1;
  const long bh = blockIdx.x;
  const int r0 = blockIdx.y * kHeadRows;
  const int rows = min(kHeadRows, ne - r0);
  const int nk = r0 + rows;  // keys visible to these rows
  float *Ks = sm;                      // [kT][dkp]
  float *Vs = Ks + kT * dkp;           // [kT][dv]
  float *Qs = Vs + kT * dv;            // [kHeadRows][dk]
  float *W = Qs + kHeadRows * dk;      // [kHeadRows][kT] weights of each row
  const int tid = threadIdx.x, nthr = kHeadRows * 32;
  const int warp = tid >> 5, lane = tid & 31;
  const Tin *qh = q + (bh * N + r0) * dk, *kh = k + bh * N * dk, *vh = v + bh * N * dv;
  // eight elements per load (rows are 16-byte aligned for the supported sizes)
  for (int e = 8 * tid; e < nk * dk; e += 8 * nthr) {
    const int t = e / dk, i = e - t * dk;
    float f[8];
    ld8(kh + e, f);
#pragma unroll
    for (int x = 0; x < 8; ++x) Ks[t * dkp + i + x] = phi(f[x]);
  }
  for (int e = 8 * tid; e < nk * dv; e += 8 * nthr) {
    float f[8];
    ld8(vh + e, f);
#pragma unroll
    for (int x = 0; x < 8; ++x) Vs[e + x] = f[x];
  }
  for (int e = 8 * tid; e < rows * dk; e += 8 * nthr) {
    float f[8];
    ld8(qh + e, f);
#pragma unroll
    for (int x = 0; x < 8; ++x) Qs[e + x] = phi(f[x]);
  }
  __syncthreads();
  if (warp >= rows) return;
  const int t = r0 + warp;  // this warp's query row
  const float *qt = Qs + warp * dk;
  float *wt = W + warp * kT;
  // weights: lane handles keys j = lane, lane + 32
  float wsum = 0.f;
  for (int j = lane; j <= t; j += 32) {
    float a = 0.f;
    for (int i = 0; i < dk; ++i) a = fmaf(qt[i], Ks[j * dkp + i], a);
    wt[j] = a;
    wsum += a;
  }
  wsum = warp_sum(wsum);
  float d = 0.f;
  if (S0) {
    for (int i = lane; i < dk; i += 32) d = fmaf(qt[i], z0[bh * dk + i], d);
    d = warp_sum(d);
  }
  const float den = (d + wsum) + eps;
  __syncwarp();
  // outputs: lane handles columns c = lane, lane + 32, ...
  const float *Sh = S0 ? S0 + bh * dk * dv : nullptr;
  for (int c = lane; c < dv; c += 32) {
    float n = 0.f;
    if (Sh)
      for (int i = 0; i < dk; ++i) n = fmaf(qt[i], Sh[i * dv + c], n);
    float m = 0.f;
    for (int j = 0; j <= t; ++j) m = fmaf(wt[j], Vs[j * dv + c], m);
    out[(bh * N + t) * dv + c] = (n + m) / den;
  }
}

template <typename Tin>
cudaError_t launch_head_t(const Problem &p, int ne, const float *S0, const float *z0) {
  const size_t smem = sizeof(float) * ((size_t)kT * (p.dk + 1) + (size_t)kT * p.dv + (size_t)kHeadRows * p.dk +
                                       (size_t)kHeadRows * kT);
  cudaError_t e = cudaFuncSetAttribute(causal_exact_head_kernel<Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  const unsigned row_blocks = (unsigned)((ne + kHeadRows - 1) / kHeadRows);
  LaunchTimer timer(kKExactHead, p.stream);
  causal_exact_head_kernel<Tin><<<dim3(p.BH, row_blocks), kHeadRows * 32, smem, p.stream>>>(
      (const Tin *)p.q, (const Tin *)p.k, (const Tin *)p.v, p.out, S0, z0, p.N, ne, p.dk, p.dv, p.eps);
  e = cudaGetLastError();
  timer.done(e);
  if (e == cudaSuccess) count_launch();
  return e;
}

}  // namespace

cudaError_t launch_causal_exact_head(const Problem &p, long n_exact, const float *S0, const float *z0) {
  if (n_exact <= 0) return cudaSuccess;
  const int ne = (int)std::min<long>(n_exact, kT);
  if (p.dt == LA_F32) return launch_head_t<float>(p, ne, S0, z0);
  return launch_head_t<__nv_bfloat16>(p, ne, S0, z0);
}

cudaError_t launch_causal_simt(const Problem &p, long n_proc, bool from_state, bool write_state) {
  if (p.dt == LA_F32) return launch_t<float>(p, n_proc, from_state, write_state);
  return launch_t<__nv_bfloat16>(p, n_proc, from_state, write_state);
}

}  // namespace la
