// One recurrent decode step per head, a pure read-modify-write of the state.
//
// S += phi(k) v^T; z += phi(k); out = phi(q)^T S / (phi(q)^T z + eps): the
// causal recurrence applied to one new token, reading the UPDATED state
// ("线性注意力从头到尾讲清楚" §7; "Linear Attention Math", "The recurrent
// form"; "Linear Attention: Accumulating KV in a Fixed-Size State": add,
// then read).  Per head the [dk, dv] fp32 state streams through registers
// once: each thread owns one float4 column quad over a strided set of rows,
// loads all of its rows before storing any (many independent 16-byte loads
// in flight), keeps its partial phi(q)^T S for those columns, and the
// partials meet in shared memory.  The state is touched exactly once per
// step, so loads and stores use the streaming (evict-first) cache hints.
//
// Retention mode (kRet): S = gamma_h S + k v^T, out = q^T S with q and k as
// given and no normalizer ("Linear Attention Math", "The kernel cousins:
// SSMs and RetNet"), the same single pass over the state.
#include "common.cuh"
#include "internal.h"

namespace la {
namespace {

constexpr int kThreads = 256;

// Per-head decays of the retention step (head bh decays by g[bh % H]).
struct Decay {
  int H;
  float g[kMaxRetentionHeads];
};

// Head sizes are template parameters: with runtime sizes the per-thread row
// loop cannot be resolved at compile time, the kernel needs ~140 registers,
// and only one CTA fits per SM, which leaves HBM a third idle.
template <typename Tin, int DK, int DV, bool kRet>
__global__ void __launch_bounds__(kThreads)
    decode_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k, const Tin *__restrict__ v,
                  float *__restrict__ out, float *__restrict__ S_g, float *__restrict__ z_g, float eps,
                  const __grid_constant__ Decay decay) {
  constexpr int kQuads = DV / 4;               // float4 column quads per row
  constexpr int kGroups = kThreads / kQuads;   // row groups
  constexpr int kRows = DK / kGroups;          // rows per thread
  static_assert(kRows >= 1 && kRows * kGroups == DK, "rows must split evenly over the row groups");
  __shared__ float fk[DK], fq[DK], vv[DV];
  __shared__ float4 part[kThreads];
  __shared__ float wden[kThreads / 32];
  const long bh = blockIdx.x;
  const int tid = threadIdx.x;
  const int cq = tid % kQuads, g = tid / kQuads;

  float4 *S4 = reinterpret_cast<float4 *>(S_g + bh * (long)DK * DV);
  float4 s[kRows];
#pragma unroll
  for (int r = 0; r < kRows; ++r) s[r] = __ldcs(S4 + (g + r * kGroups) * kQuads + cq);

  // normalizer first (its loads overlap the state's): z += phi(k), den = phi(q) . z_new
  float d = 0.f;
  if (tid < DK) {
    if (kRet) {
      fk[tid] = ldf(k + bh * DK + tid);
      fq[tid] = ldf(q + bh * DK + tid);
    } else {
      const float a = phi(ldf(k + bh * DK + tid)), b = phi(ldf(q + bh * DK + tid));
      const float zn = z_g[bh * DK + tid] + a;
      fk[tid] = a;
      fq[tid] = b;
      z_g[bh * DK + tid] = zn;
      d = b * zn;
    }
  }
  if (tid < DV) vv[tid] = ldf(v + bh * DV + tid);
  d = warp_sum(d);
  if ((tid & 31) == 0) wden[tid >> 5] = d;
  __syncthreads();

  const float4 vq = reinterpret_cast<const float4 *>(vv)[cq];
  const float gam = kRet ? decay.g[bh % decay.H] : 1.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int r = 0; r < kRows; ++r) {
    const int i = g + r * kGroups;
    const float a = fk[i], b = fq[i];
    float4 x = s[r];
    if (kRet) x = make_float4(gam * x.x, gam * x.y, gam * x.z, gam * x.w);
    x.x = fmaf(a, vq.x, x.x);
    x.y = fmaf(a, vq.y, x.y);
    x.z = fmaf(a, vq.z, x.z);
    x.w = fmaf(a, vq.w, x.w);
    __stcs(S4 + i * kQuads + cq, x);
    acc.x = fmaf(b, x.x, acc.x);
    acc.y = fmaf(b, x.y, acc.y);
    acc.z = fmaf(b, x.z, acc.z);
    acc.w = fmaf(b, x.w, acc.w);
  }
  part[g * kQuads + cq] = acc;
  __syncthreads();
  if (tid < DV) {
    float den = 0.f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) den += wden[w];
    const float *pf = reinterpret_cast<const float *>(part);
    float num = 0.f;
#pragma unroll
    for (int gg = 0; gg < kGroups; ++gg) num += pf[gg * DV + tid];
    out[bh * DV + tid] = kRet ? num : num / (den + eps);
  }
}

template <typename Tin, int DK, int DV>
cudaError_t launch_t(const Problem &p, const Decay *decay) {
  LaunchTimer timer(decay ? kKRetentionDecode : kKDecode, p.stream);
  Decay none;
  none.H = 1;
  none.g[0] = 1.f;
  if (decay)
    decode_kernel<Tin, DK, DV, true><<<p.BH, kThreads, 0, p.stream>>>(
        (const Tin *)p.q, (const Tin *)p.k, (const Tin *)p.v, p.out, p.S, nullptr, 0.f, *decay);
  else
    decode_kernel<Tin, DK, DV, false><<<p.BH, kThreads, 0, p.stream>>>(
        (const Tin *)p.q, (const Tin *)p.k, (const Tin *)p.v, p.out, p.S, p.z, p.eps, none);
  const cudaError_t e = cudaGetLastError();
  timer.done(e);
  if (e == cudaSuccess) count_launch();
  return e;
}

template <typename Tin, int DK>
cudaError_t launch_dv(const Problem &p, const Decay *decay) {
  if (p.dv == 32) return launch_t<Tin, DK, 32>(p, decay);
  if (p.dv == 64) return launch_t<Tin, DK, 64>(p, decay);
  return launch_t<Tin, DK, 128>(p, decay);
}

template <typename Tin>
cudaError_t launch_dk(const Problem &p, const Decay *decay) {
  if (p.dk == 32) return launch_dv<Tin, 32>(p, decay);
  if (p.dk == 64) return launch_dv<Tin, 64>(p, decay);
  return launch_dv<Tin, 128>(p, decay);
}

cudaError_t launch_any(const Problem &p, const Decay *decay) {
  if (p.dt == LA_F32) return launch_dk<float>(p, decay);
  return launch_dk<__nv_bfloat16>(p, decay);
}

}  // namespace

cudaError_t launch_decode(const Problem &p) { return launch_any(p, nullptr); }

cudaError_t launch_retention_decode(const Problem &p, const float *gamma, int H) {
  if (!gamma || H < 1 || H > kMaxRetentionHeads) return cudaErrorInvalidValue;
  Decay d;
  d.H = H;
  for (int h = 0; h < kMaxRetentionHeads; ++h) d.g[h] = h < H ? gamma[h] : 1.f;
  return launch_any(p, &d);
}

}  // namespace la
