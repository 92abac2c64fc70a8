// Gradient of the causal prefill on CUDA cores, exact fp32.
//
// The forward is o_t = phi(q_t)^T S_t / (phi(q_t)^T z_t + eps) with the
// state inclusive of token t ("线性注意力从头到尾讲清楚" §7; "Linear Attention
// Math", "The recurrent form").  The pages name training through the chunked
// form ("Linear Attention: From Pairwise Reads to a Recurrent State", "A
// recurrence need not force token-serial training") but write no backward
// pass; this is the derivative of that definition.  With the upstream
// gradient dO_t,
//   gnum_t = dO_t / den_t,  gden_t = -(dO_t . o_t) / den_t,
//   dphi(q_t) = S_t gnum_t + z_t gden_t,
//   dphi(k_j) = U_j v_j + u_j,  dv_j = U_j^T phi(k_j),
// where U_j = dS_N + sum_{t >= j} phi(q_t) gnum_t^T and
// u_j = dz_N + sum_{t >= j} phi(q_t) gden_t; the initial state's gradient is
// (U_0, u_0).  phi = ELU + 1 gives phi'(x) = min(phi(x), 1), so only phi of
// the inputs is kept.
//
// One CTA per head, 64-token chunks, all arithmetic in fp32:
//   pass 1 (chunks in order): the state S, z; per chunk the masked scores
//     A = tril(phi(Q) phi(K)^T), the denominators, the outputs, gnum and
//     gden (kept in a scratch row per token), and dq;
//   pass 2 (chunks in reverse): U, u in place of S, z; per chunk dk and dv
//     from the carried U, u and the chunk's own masked terms.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace la {
namespace {

constexpr int kT = 64;  // tokens per chunk
constexpr int kThreads = 256;

size_t bwd_smem_bytes(int dk, int dv) {
  const size_t dkp = dk + 1, dvp = dv + 1;
  return sizeof(float) * ((size_t)dk * dvp + dk + 2 * kT * dkp + kT * dvp + (size_t)kT * dv + 2 * (size_t)kT * (kT + 1) +
                          2 * kT);
}

template <typename Tin>
__global__ void __launch_bounds__(kThreads)
    causal_backward_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k, const Tin *__restrict__ v,
                           const float *__restrict__ dout, const float *__restrict__ S0,
                           const float *__restrict__ z0, const float *__restrict__ dSN,
                           const float *__restrict__ dzN, float *__restrict__ dq, float *__restrict__ dk_g,
                           float *__restrict__ dv_g, float *__restrict__ dS0, float *__restrict__ dz0,
                           float *__restrict__ G, long N, int dk, int dv, float eps) {
  extern __shared__ float sm[];
  // padded rows (dk + 1, dv + 1): lanes that walk consecutive rows hit distinct banks
  const int dkp = dk + 1, dvp = dv + 1;
  float *S = sm;                   // [dk][dvp] state (pass 1), U (pass 2)
  float *z = S + dk * dvp;         // [dk]      normalizer (pass 1), u (pass 2)
  float *Qs = z + dk;              // [kT][dkp] phi(q)
  float *Ks = Qs + kT * dkp;       // [kT][dkp] phi(k)
  float *Vs = Ks + kT * dkp;       // [kT][dvp] v
  float *Gs = Vs + kT * dvp;       // [kT][dv]  dO, then gnum
  float *A = Gs + kT * dv;         // [kT][kT+1] phi(q_t).phi(k_j), j <= t
  float *Bm = A + kT * (kT + 1);   // [kT][kT+1] v_j.gnum_t + gden_t, j <= t
  float *den = Bm + kT * (kT + 1); // [kT]
  float *gd = den + kT;            // [kT] gden

  const long bh = blockIdx.x;
  const int tid = threadIdx.x;
  const Tin *qh = q + bh * N * dk, *kh = k + bh * N * dk, *vh = v + bh * N * dv;
  const float *oh = dout + bh * N * dv;
  float *dqh = dq + bh * N * dk, *dkh = dk_g + bh * N * dk, *dvh = dv_g + bh * N * dv;
  float *Gh = G + bh * N * (dv + 1);  // per token: gnum (dv), gden

  for (int e = tid; e < dk * dv; e += kThreads) S[(e / dv) * dvp + e % dv] = S0 ? S0[bh * dk * dv + e] : 0.f;
  for (int i = tid; i < dk; i += kThreads) z[i] = z0 ? z0[bh * dk + i] : 0.f;

  // ---------------- pass 1: chunks in order ----------------
  for (long t0 = 0; t0 < N; t0 += kT) {
    const int T = (int)min((long)kT, N - t0);
    __syncthreads();  // the previous chunk is fully consumed
    for (int e = tid; e < T * dk; e += kThreads) {
      const int t = e / dk, i = e - t * dk;
      Qs[t * dkp + i] = phi(ldf(qh + (t0 + t) * dk + i));
      Ks[t * dkp + i] = phi(ldf(kh + (t0 + t) * dk + i));
    }
    for (int e = tid; e < T * dv; e += kThreads) {
      Vs[(e / dv) * dvp + e % dv] = ldf(vh + t0 * dv + e);
      Gs[e] = oh[t0 * dv + e];
    }
    __syncthreads();
    for (int e = tid; e < T * T; e += kThreads) {
      const int t = e / T, j = e - t * T;
      float a = 0.f;
      if (j <= t)
        for (int i = 0; i < dk; ++i) a = fmaf(Qs[t * dkp + i], Ks[j * dkp + i], a);
      A[t * (kT + 1) + j] = a;
    }
    __syncthreads();
    for (int t = tid; t < T; t += kThreads) {
      float d = 0.f;
      for (int i = 0; i < dk; ++i) d = fmaf(Qs[t * dkp + i], z[i], d);
      float a = 0.f;
      for (int j = 0; j <= t; ++j) a += A[t * (kT + 1) + j];
      den[t] = (d + a) + eps;
    }
    __syncthreads();
    // outputs o_t (recomputed), dO_t . o_t per row by one warp each
    {
      const int warp = tid >> 5, lane = tid & 31;
      for (int t = warp; t < T; t += kThreads / 32) {
        float dot = 0.f;
        for (int c = lane; c < dv; c += 32) {
          float n = 0.f;
#pragma unroll 8
          for (int i = 0; i < dk; ++i) n = fmaf(Qs[t * dkp + i], S[i * dvp + c], n);
          for (int j = 0; j <= t; ++j) n = fmaf(A[t * (kT + 1) + j], Vs[j * dvp + c], n);
          dot = fmaf(Gs[t * dv + c], n / den[t], dot);
        }
        dot = warp_sum(dot);
        if (lane == 0) gd[t] = -dot / den[t];
      }
    }
    __syncthreads();
    for (int e = tid; e < T * dv; e += kThreads) {
      const int t = e / dv;
      Gs[e] /= den[t];  // gnum
    }
    __syncthreads();
    // B_tj = v_j . gnum_t + gden_t (j <= t); the scratch rows of gnum and gden
    for (int e = tid; e < T * T; e += kThreads) {
      const int t = e / T, j = e - t * T;
      float b = 0.f;
      if (j <= t) {
#pragma unroll 8
        for (int c = 0; c < dv; ++c) b = fmaf(Vs[j * dvp + c], Gs[t * dv + c], b);
        b += gd[t];
      }
      Bm[t * (kT + 1) + j] = b;
    }
    for (int e = tid; e < T * (dv + 1); e += kThreads) {
      const int t = e / (dv + 1), c = e - t * (dv + 1);
      Gh[(t0 + t) * (dv + 1) + c] = c < dv ? Gs[t * dv + c] : gd[t];
    }
    __syncthreads();
    // dphi(q_t) = S_prev gnum_t + z_prev gden_t + sum_{j <= t} B_tj phi(k_j)
    for (int e = tid; e < T * dk; e += kThreads) {
      const int t = e / dk, i = e - t * dk;
      float g = z[i] * gd[t];
#pragma unroll 8
      for (int c = 0; c < dv; ++c) g = fmaf(S[i * dvp + c], Gs[t * dv + c], g);
      for (int j = 0; j <= t; ++j) g = fmaf(Bm[t * (kT + 1) + j], Ks[j * dkp + i], g);
      dqh[(t0 + t) * dk + i] = g * fminf(Qs[t * dkp + i], 1.f);
    }
    __syncthreads();
    // fold the chunk into the state
    for (int e = tid; e < dk * dv; e += kThreads) {
      const int i = e / dv, c = e - i * dv;
      float s = 0.f;
#pragma unroll 8
      for (int j = 0; j < T; ++j) s = fmaf(Ks[j * dkp + i], Vs[j * dvp + c], s);
      S[i * dvp + c] += s;
    }
    for (int i = tid; i < dk; i += kThreads) {
      float s = 0.f;
      for (int j = 0; j < T; ++j) s += Ks[j * dkp + i];
      z[i] += s;
    }
  }

  // ---------------- pass 2: chunks in reverse ----------------
  __syncthreads();
  for (int e = tid; e < dk * dv; e += kThreads) S[(e / dv) * dvp + e % dv] = dSN ? dSN[bh * dk * dv + e] : 0.f;  // U
  for (int i = tid; i < dk; i += kThreads) z[i] = dzN ? dzN[bh * dk + i] : 0.f;            // u
  const long nch = (N + kT - 1) / kT;
  for (long ci = nch - 1; ci >= 0; --ci) {
    const long t0 = ci * kT;
    const int T = (int)min((long)kT, N - t0);
    __syncthreads();
    for (int e = tid; e < T * dk; e += kThreads) {
      const int t = e / dk, i = e - t * dk;
      Qs[t * dkp + i] = phi(ldf(qh + (t0 + t) * dk + i));
      Ks[t * dkp + i] = phi(ldf(kh + (t0 + t) * dk + i));
    }
    for (int e = tid; e < T * dv; e += kThreads) {
      const int t = e / dv, c = e - t * dv;
      Vs[t * dvp + c] = ldf(vh + t0 * dv + e);
      Gs[e] = Gh[(t0 + t) * (dv + 1) + c];
    }
    for (int t = tid; t < T; t += kThreads) gd[t] = Gh[(t0 + t) * (dv + 1) + dv];
    __syncthreads();
    for (int e = tid; e < T * T; e += kThreads) {
      const int t = e / T, j = e - t * T;
      float a = 0.f, b = 0.f;
      if (j <= t) {
#pragma unroll 8
        for (int i = 0; i < dk; ++i) a = fmaf(Qs[t * dkp + i], Ks[j * dkp + i], a);
#pragma unroll 8
        for (int c = 0; c < dv; ++c) b = fmaf(Vs[j * dvp + c], Gs[t * dv + c], b);
        b += gd[t];
      }
      A[t * (kT + 1) + j] = a;
      Bm[t * (kT + 1) + j] = b;
    }
    __syncthreads();
    // dphi(k_j) = U v_j + u + sum_{t >= j} B_tj phi(q_t)
    for (int e = tid; e < T * dk; e += kThreads) {
      const int j = e / dk, i = e - j * dk;
      float g = z[i];
#pragma unroll 8
      for (int c = 0; c < dv; ++c) g = fmaf(S[i * dvp + c], Vs[j * dvp + c], g);
      for (int t = j; t < T; ++t) g = fmaf(Bm[t * (kT + 1) + j], Qs[t * dkp + i], g);
      dkh[(t0 + j) * dk + i] = g * fminf(Ks[j * dkp + i], 1.f);
    }
    // dv_j = U^T phi(k_j) + sum_{t >= j} A_tj gnum_t
    for (int e = tid; e < T * dv; e += kThreads) {
      const int j = e / dv, c = e - j * dv;
      float g = 0.f;
#pragma unroll 8
      for (int i = 0; i < dk; ++i) g = fmaf(S[i * dvp + c], Ks[j * dkp + i], g);
      for (int t = j; t < T; ++t) g = fmaf(A[t * (kT + 1) + j], Gs[t * dv + c], g);
      dvh[(t0 + j) * dv + c] = g;
    }
    __syncthreads();
    // U += sum_t phi(q_t) gnum_t^T, u += sum_t phi(q_t) gden_t
    for (int e = tid; e < dk * dv; e += kThreads) {
      const int i = e / dv, c = e - i * dv;
      float s = 0.f;
#pragma unroll 8
      for (int t = 0; t < T; ++t) s = fmaf(Qs[t * dkp + i], Gs[t * dv + c], s);
      S[i * dvp + c] += s;
    }
    for (int i = tid; i < dk; i += kThreads) {
      float s = 0.f;
      for (int t = 0; t < T; ++t) s = fmaf(Qs[t * dkp + i], gd[t], s);
      z[i] += s;
    }
  }
  __syncthreads();
  if (dS0)
    for (int e = tid; e < dk * dv; e += kThreads) dS0[bh * dk * dv + e] = S[(e / dv) * dvp + e % dv];
  if (dz0)
    for (int i = tid; i < dk; i += kThreads) dz0[bh * dk + i] = z[i];
}

template <typename Tin>
cudaError_t launch_t(const BackwardProblem &b, float *G) {
  const Problem &p = b.p;
  const size_t smem = bwd_smem_bytes(p.dk, p.dv);
  cudaError_t e = cudaFuncSetAttribute(causal_backward_kernel<Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  LaunchTimer timer(kKBackward, p.stream);
  causal_backward_kernel<Tin><<<p.BH, kThreads, smem, p.stream>>>(
      (const Tin *)p.q, (const Tin *)p.k, (const Tin *)p.v, b.dout, b.S0, b.z0, b.dS, b.dz, b.dq, b.dk, b.dv,
      b.dS0, b.dz0, G, p.N, p.dk, p.dv, p.eps);
  e = cudaGetLastError();
  timer.done(e);
  if (e == cudaSuccess) count_launch();
  return e;
}

}  // namespace

cudaError_t launch_causal_backward(const BackwardProblem &b) {
  const Problem &p = b.p;
  // scratch: gnum and gden of every token, written by pass 1 and read by pass 2
  const size_t g_bytes = sizeof(float) * (size_t)p.BH * p.N * (p.dv + 1);
  float *G = nullptr;
  cudaError_t e = cudaMallocAsync(reinterpret_cast<void **>(&G), std::max<size_t>(g_bytes, 16), p.stream);
  if (e != cudaSuccess) return e;
  e = p.dt == LA_F32 ? launch_t<float>(b, G) : launch_t<__nv_bfloat16>(b, G);
  const cudaError_t f = cudaFreeAsync(G, p.stream);
  return e != cudaSuccess ? e : f;
}

}  // namespace la
