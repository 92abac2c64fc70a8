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
#include "common.cuh"
#include "internal.h"

namespace la {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxRows = 16;  // rows per thread: dk * dv / (4 * kThreads) <= 16

template <typename Tin>
__global__ void __launch_bounds__(kThreads)
    decode_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k, const Tin *__restrict__ v,
                  float *__restrict__ out, float *__restrict__ S_g, float *__restrict__ z_g, int dk,
                  int dv, float eps) {
  __shared__ float fk[128], fq[128], vv[128];
  __shared__ float part[kThreads * 4];
  __shared__ float wden[kThreads / 32];
  const long bh = blockIdx.x;
  const int tid = threadIdx.x;
  const int nq = dv >> 2;           // float4 column quads per row
  const int groups = kThreads / nq; // row groups
  const int cq = tid % nq, g = tid / nq;
  const int nr = dk / groups;       // rows per thread

  float4 *S4 = reinterpret_cast<float4 *>(S_g + bh * (long)dk * dv);
  float4 s[kMaxRows];
#pragma unroll
  for (int r = 0; r < kMaxRows; ++r)
    if (r < nr) s[r] = __ldcs(S4 + (long)(g + r * groups) * nq + cq);

  if (tid < dk) {
    fk[tid] = phi(ldf(k + bh * dk + tid));
    fq[tid] = phi(ldf(q + bh * dk + tid));
  }
  if (tid < dv) vv[tid] = ldf(v + bh * dv + tid);
  __syncthreads();

  const float4 vq = make_float4(vv[4 * cq], vv[4 * cq + 1], vv[4 * cq + 2], vv[4 * cq + 3]);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int r = 0; r < kMaxRows; ++r) {
    if (r < nr) {
      const int i = g + r * groups;
      const float a = fk[i], b = fq[i];
      float4 x = s[r];
      x.x = fmaf(a, vq.x, x.x);
      x.y = fmaf(a, vq.y, x.y);
      x.z = fmaf(a, vq.z, x.z);
      x.w = fmaf(a, vq.w, x.w);
      __stcs(S4 + (long)i * nq + cq, x);
      acc.x = fmaf(b, x.x, acc.x);
      acc.y = fmaf(b, x.y, acc.y);
      acc.z = fmaf(b, x.z, acc.z);
      acc.w = fmaf(b, x.w, acc.w);
    }
  }
  reinterpret_cast<float4 *>(part)[g * nq + cq] = acc;

  // normalizer: z += phi(k), den = phi(q) . z_new
  float d = 0.f;
  if (tid < dk) {
    const float zn = z_g[bh * dk + tid] + fk[tid];
    z_g[bh * dk + tid] = zn;
    d = fq[tid] * zn;
  }
  d = warp_sum(d);
  if ((tid & 31) == 0) wden[tid >> 5] = d;
  __syncthreads();
  if (tid < dv) {
    float den = 0.f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) den += wden[w];
    float num = 0.f;
    for (int gg = 0; gg < groups; ++gg) num += part[gg * dv + tid];
    out[bh * dv + tid] = num / (den + eps);
  }
}

template <typename Tin>
cudaError_t launch_t(const Problem &p) {
  decode_kernel<Tin><<<p.BH, kThreads, 0, p.stream>>>((const Tin *)p.q, (const Tin *)p.k, (const Tin *)p.v, p.out,
                                                    p.S, p.z, p.dk, p.dv, p.eps);
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) count_launch();
  return e;
}

}  // namespace

cudaError_t launch_decode(const Problem &p) {
  if (p.dt == LA_F32) return launch_t<float>(p);
  return launch_t<__nv_bfloat16>(p);
}

}  // namespace la
