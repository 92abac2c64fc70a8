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

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace la {
namespace {

constexpr int kThreads = 256;

// Shared memory of a chunk length kT: the state, z, phi(Q) and phi(K) rows (padded), V, the
// masked weights and the denominators.
size_t simt_smem_bytes(int dk, int dv, int kT) {
  const size_t floats = (size_t)dk * dv + dk + 2 * (size_t)kT * (dk + 1) + (size_t)kT * dv +
                        (size_t)kT * (kT + 1) + kT;
  return floats * sizeof(float);
}

// kT: tokens per chunk, 64, or 32 where the state is too large for 64 (256 given features).
template <typename Tin, int kT>
__global__ void __launch_bounds__(kThreads)
    causal_simt_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k, const Tin *__restrict__ v,
                       float *__restrict__ out, float *__restrict__ S_g, float *__restrict__ z_g,
                       long N, long n_proc, int dk, int dv, float eps, int from_state,
                       int write_state, int identity) {
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
      const float xq = ldf(qh + (t0 + t) * dk + i), xk = ldf(kh + (t0 + t) * dk + i);
      Qs[t * dkp + i] = identity ? xq : phi(xq);  // identity: q and k are given features
      Ks[t * dkp + i] = identity ? xk : phi(xk);
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

template <typename Tin, int kT>
cudaError_t launch_t(const Problem &p, long n_proc, bool from_state, bool write_state, bool identity) {
  const size_t smem = simt_smem_bytes(p.dk, p.dv, kT);
  cudaError_t e = cudaFuncSetAttribute(causal_simt_kernel<Tin, kT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  LaunchTimer timer(kKCausalSimt, p.stream);
  causal_simt_kernel<Tin, kT><<<p.BH, kThreads, smem, p.stream>>>(
      (const Tin *)p.q, (const Tin *)p.k, (const Tin *)p.v, p.out, p.S, p.z, p.N, n_proc, p.dk, p.dv, p.eps,
      from_state ? 1 : 0, write_state ? 1 : 0, identity ? 1 : 0);
  e = cudaGetLastError();
  timer.done(e);
  if (e == cudaSuccess) count_launch();
  return e;
}

// Exact fp32 outputs for tokens [0, ne) of a head (ne <= 64).  The leading
// tokens of a sequence read a state built from few tokens, so their outputs
// are O(1) while later ones average down; they get full fp32 weights here
// instead of the tensor cores' bf16 operands.  One CTA per head: phi(Q),
// phi(K) and V of the leading rows are staged in fp32, the masked weights
// W = tril(phi(Q) phi(K)^T) and the outputs W V (plus phi(Q) S0 and
// phi(Q).z0 for a carried state) are formed with register micro-tiles, and
// every row is divided by its own denominator sum_j W_tj (+ phi(q_t).z0) + eps.
constexpr int kHeadThreads = 256;
constexpr int kHeadMax = 64;

template <int DK, int DV>
struct HeadSmem {
  static constexpr int P = DK + 1;  // padded rows of phi(Q), phi(K): column reads conflict-free
  static constexpr int WP = kHeadMax + 1;
  static constexpr size_t Bytes = sizeof(float) * ((size_t)2 * kHeadMax * P + kHeadMax * DV + kHeadMax * WP + kHeadMax);
  // the caller's state, once the keys and values are done with, over phi(K) and V (contiguous)
  static_assert((size_t)kHeadMax * P + kHeadMax * DV >= (size_t)DK * DV, "the state fits over phi(K) and V");
};

template <typename Tin, int DK, int DV>
__global__ void __launch_bounds__(kHeadThreads)
    causal_exact_head_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k, const Tin *__restrict__ v,
                             float *__restrict__ out, const float *__restrict__ S0, const float *__restrict__ z0,
                             long N, int ne, float eps) {
  using L = HeadSmem<DK, DV>;
  constexpr int P = L::P, WP = L::WP;
  extern __shared__ float sm[];
  float *Qf = sm, *Kf = Qf + kHeadMax * P, *Vf = Kf + kHeadMax * P, *W = Vf + kHeadMax * DV, *den = W + kHeadMax * WP;
  const long bh = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const Tin *qh = q + bh * N * DK, *kh = k + bh * N * DK, *vh = v + bh * N * DV;
  // stage rows [0, ne) in fp32 (eight elements per 16-byte-aligned load); rows past ne are zero
  for (int e = 8 * tid; e < kHeadMax * DK; e += 8 * kHeadThreads) {
    const int t = e / DK, i = e % DK;
    float fq[8], fk[8];
    if (t < ne) {
      ld8(qh + e, fq);
      ld8(kh + e, fk);
    }
#pragma unroll
    for (int x = 0; x < 8; ++x) {
      Qf[t * P + i + x] = t < ne ? phi(fq[x]) : 0.f;
      Kf[t * P + i + x] = t < ne ? phi(fk[x]) : 0.f;
    }
  }
  for (int e = 8 * tid; e < kHeadMax * DV; e += 8 * kHeadThreads) {
    const int t = e / DV;
    float f[8];
    if (t < ne) ld8(vh + e, f);
#pragma unroll
    for (int x = 0; x < 8; ++x) Vf[e + x] = t < ne ? f[x] : 0.f;
  }
  __syncthreads();
  {
    // W: thread (ty, tx) forms rows ty + 16 r and keys tx + 16 c, r, c < 4
    const int ty = tid >> 4, tx = tid & 15;
    float a[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) a[r][c] = 0.f;
#pragma unroll 4
    for (int i = 0; i < DK; ++i) {
      float qv[4], kv[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) qv[r] = Qf[(ty + 16 * r) * P + i];
#pragma unroll
      for (int c = 0; c < 4; ++c) kv[c] = Kf[(tx + 16 * c) * P + i];
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) a[r][c] = fmaf(qv[r], kv[c], a[r][c]);
    }
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int i = ty + 16 * r, j = tx + 16 * c;
        W[i * WP + j] = j <= i ? a[r][c] : 0.f;  // inclusive causal mask
      }
  }
  __syncthreads();
  // denominators, one warp per row at a time
  for (int i = warp; i < kHeadMax; i += kHeadThreads / 32) {
    float s = W[i * WP + lane] + W[i * WP + lane + 32];
    if (z0)
      for (int f = lane; f < DK; f += 32) s = fmaf(Qf[i * P + f], z0[bh * DK + f], s);
    s = warp_sum(s);
    if (lane == 0) den[i] = s + eps;
  }
  __syncthreads();
  {
    // outputs: warp w takes rows 8w .. 8w + 7, lane the columns lane + 32 c
    constexpr int kCols = DV / 32;
    const int r0 = 8 * warp;
    float o[8][kCols];
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
      for (int c = 0; c < kCols; ++c) o[r][c] = 0.f;
    const int jmax = min(ne, r0 + 8);  // keys visible to the last of these rows
    for (int j = 0; j < jmax; ++j) {
      float vv[kCols];
#pragma unroll
      for (int c = 0; c < kCols; ++c) vv[c] = Vf[j * DV + lane + 32 * c];
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const float w = W[(r0 + r) * WP + j];
#pragma unroll
        for (int c = 0; c < kCols; ++c) o[r][c] = fmaf(w, vv[c], o[r][c]);
      }
    }
    if (S0) {
      // stage the caller's state over phi(K) and V (every read of those is done), all loads in flight
      float *Sh = Kf;
      __syncthreads();
      const float4 *src = reinterpret_cast<const float4 *>(S0 + bh * DK * DV);
      for (int e = tid; e < DK * DV / 4; e += kHeadThreads) reinterpret_cast<float4 *>(Sh)[e] = src[e];
      __syncthreads();
      for (int f = 0; f < DK; ++f) {
        float sv[kCols];
#pragma unroll
        for (int c = 0; c < kCols; ++c) sv[c] = Sh[f * DV + lane + 32 * c];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const float qf = Qf[(r0 + r) * P + f];
#pragma unroll
          for (int c = 0; c < kCols; ++c) o[r][c] = fmaf(qf, sv[c], o[r][c]);
        }
      }
    }
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int t = r0 + r;
      if (t < ne)
#pragma unroll
        for (int c = 0; c < kCols; ++c) out[(bh * N + t) * DV + lane + 32 * c] = o[r][c] / den[t];
    }
  }
  // When launched early beside the previous kernel of the stream, this grid
  // completes only after that kernel: the last CTA waits for it.
  if (blockIdx.x == gridDim.x - 1) asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <typename Tin, int DK, int DV>
cudaError_t launch_head_t(const Problem &p, int ne, const float *S0, const float *z0, bool pdl) {
  const cudaError_t attr =
      ensure_smem_optin((const void *)causal_exact_head_kernel<Tin, DK, DV>, (int)HeadSmem<DK, DV>::Bytes);
  if (attr != cudaSuccess) return attr;
  LaunchTimer timer(kKExactHead, p.stream);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute early[1];
  early[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  early[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3((unsigned)p.BH);
  cfg.blockDim = dim3(kHeadThreads);
  cfg.dynamicSmemBytes = HeadSmem<DK, DV>::Bytes;
  cfg.stream = p.stream;
  cfg.attrs = early;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, causal_exact_head_kernel<Tin, DK, DV>, (const Tin *)p.q, (const Tin *)p.k,
                                     (const Tin *)p.v, p.out, S0, z0, p.N, ne, p.eps);
  if (e == cudaSuccess) e = cudaGetLastError();
  timer.done(e);
  if (e == cudaSuccess) count_launch();
  return e;
}

}  // namespace

cudaError_t launch_causal_exact_head(const Problem &p, long n_exact, const float *S0, const float *z0, bool pdl) {
  if (n_exact <= 0) return cudaSuccess;
  if (p.dk != 128 || p.dv != 128) return cudaErrorInvalidValue;  // serves the d = 128 tensor-core pass
  const int ne = (int)std::min<long>(n_exact, kHeadMax);
  if (p.dt == LA_F32) return launch_head_t<float, 128, 128>(p, ne, S0, z0, pdl);
  return launch_head_t<__nv_bfloat16, 128, 128>(p, ne, S0, z0, pdl);
}

cudaError_t launch_causal_simt(const Problem &p, long n_proc, bool from_state, bool write_state, bool identity) {
  // 64-token chunks where they fit the device's shared memory, else 32 (a 256 x 128 state)
  const size_t optin = (size_t)device_info(-1).max_smem_optin;
  const bool wide = simt_smem_bytes(p.dk, p.dv, 64) > optin;
  if (wide && simt_smem_bytes(p.dk, p.dv, 32) > optin) return cudaErrorInvalidValue;
  if (p.dt == LA_F32)
    return wide ? launch_t<float, 32>(p, n_proc, from_state, write_state, identity)
                : launch_t<float, 64>(p, n_proc, from_state, write_state, identity);
  return wide ? launch_t<__nv_bfloat16, 32>(p, n_proc, from_state, write_state, identity)
              : launch_t<__nv_bfloat16, 64>(p, n_proc, from_state, write_state, identity);
}

}  // namespace la
