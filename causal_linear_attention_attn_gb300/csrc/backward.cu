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
// 64-token chunks, all arithmetic in fp32.  Each head's sequence is cut into
// segments, one CTA per (segment, head), and a call runs four phases of one
// kernel template:
//   segment sums: phi(K)^T V and colsum phi(K) of every segment but the last,
//     each segment in parts with a CTA each;
//   pass 1 (chunks in order from S0 plus the earlier segments' part sums):
//     the state S, z; per chunk the masked scores A = tril(phi(Q) phi(K)^T),
//     the denominators, gnum and gden, and dq.  The outputs themselves are
//     never formed: with Y = dO S_prev^T and C = dO V^T,
//     dO_t . o_t = (phi(q_t) . Y_t + sum_j A_tj C_tj) / den_t, and Y_t / den_t
//     is dq's state term.  gnum, gden, A and the score gradients
//     Bm = tril(C / den + gden) go to scratch for pass 2;
//   gradient sums: phi(Q)^T gnum and phi(Q)^T gden of every segment but the
//     first, in parts;
//   pass 2 (chunks in reverse from dS plus the later segments' part sums):
//     U, u in place of S, z; per chunk dk and dv from the carried U, u and
//     pass 1's A and Bm; the first segment's final U, u are the initial
//     state's gradient.
// Every product is a small matrix product over shared-memory operands: the
// 256 threads form a 16 x 16 grid and thread (ty, tx) accumulates the rows
// ty + 16 r (or, where an operand is triangular, the rows 4 ty .. 4 ty + 3,
// so that its k loop stops at the diagonal) and the columns tx + 16 c of the
// result in registers.  Rows of phi(Q), phi(K), V and S are padded by one
// float so that lanes walking consecutive rows hit distinct banks.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace la {
namespace {

constexpr int kT = 64;          // tokens per chunk
constexpr int kThreads = 256;   // a 16 x 16 grid of threads
static_assert(kThreads >= 64, "one thread per token of a chunk");

template <int DK, int DV>
struct BwdSmem {
  static constexpr int KP = DK + 1, VP = DV + 1, AP = kT + 1;  // padded row lengths
  static constexpr size_t Floats =
      (size_t)DK * VP + DK + 2 * (size_t)kT * KP + (size_t)kT * VP + (size_t)kT * DV + 2 * (size_t)kT * AP + 2 * kT;
  static constexpr size_t Bytes = Floats * sizeof(float);
};
static_assert(BwdSmem<128, 128>::Bytes <= 232448, "shared memory budget");

// acc[r][c] += sum_{k0 <= k < k1} a(row(r), k) b(k, tx + 16 c), where row(r) is ty + 16 r,
// or TR ty + r with kBlockRows (each thread's rows consecutive, so that a triangular
// operand bounds its k range); pairs of columns share one packed fp32 FMA (TC is even)
template <int TR, int TC, bool kBlockRows = false, typename FA, typename FB>
__device__ __forceinline__ void tile_fma(float (&acc)[TR][TC], int k0, int k1, int ty, int tx, FA a, FB b) {
  static_assert(TC % 2 == 0, "columns go in pairs");
#pragma unroll 4
  for (int k = k0; k < k1; ++k) {
    float av[TR], bv[TC];
#pragma unroll
    for (int r = 0; r < TR; ++r) av[r] = a(kBlockRows ? TR * ty + r : ty + 16 * r, k);
#pragma unroll
    for (int c = 0; c < TC; ++c) bv[c] = b(k, tx + 16 * c);
#pragma unroll
    for (int r = 0; r < TR; ++r)
#pragma unroll
      for (int c = 0; c < TC; c += 2) {
        const float2 y = __ffma2_rn(make_float2(av[r], av[r]), make_float2(bv[c], bv[c + 1]),
                                    make_float2(acc[r][c], acc[r][c + 1]));
        acc[r][c] = y.x;
        acc[r][c + 1] = y.y;
      }
  }
}

template <int TR, int TC, typename FA, typename FB>
__device__ __forceinline__ void tile_fma(float (&acc)[TR][TC], int K, int ty, int tx, FA a, FB b) {
  tile_fma<TR, TC, false>(acc, 0, K, ty, tx, a, b);
}

// Eight consecutive inputs as loaded by one 16-byte (bf16) or two 16-byte (fp32) loads.
template <typename T>
struct Raw8;
template <>
struct Raw8<__nv_bfloat16> {
  uint4 u;
  __device__ __forceinline__ void load(const __nv_bfloat16 *p) { u = __ldg(reinterpret_cast<const uint4 *>(p)); }
  __device__ __forceinline__ float operator[](int e) const {
    const uint32_t w = e < 2 ? u.x : e < 4 ? u.y : e < 6 ? u.z : u.w;
    return __uint_as_float(e & 1 ? (w & 0xffff0000u) : (w << 16));  // bf16 is the top half of an fp32
  }
};
template <>
struct Raw8<float> {
  float4 a, b;
  __device__ __forceinline__ void load(const float *p) {
    a = __ldg(reinterpret_cast<const float4 *>(p));
    b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
  }
  __device__ __forceinline__ float operator[](int e) const {
    return e < 4 ? (e < 2 ? (e ? a.y : a.x) : (e == 2 ? a.z : a.w)) : (e < 6 ? (e == 4 ? b.x : b.y) : (e == 6 ? b.z : b.w));
  }
};

// One chunk's rows [0, T) of a row-major [*][W] block, staged in two steps so
// that the loads of several blocks are all in flight before any is stored:
// load() issues 16-byte loads (the C ABI requires 16-byte aligned inputs, and
// every chunk of a head starts at a multiple of 64 rows), store() writes f(x)
// into shared memory rows of P floats.
template <int W, typename T>
struct ChunkRows {
  static constexpr int kIt = kT * W / (8 * kThreads);
  static_assert(kIt >= 1 && kT * W % (8 * kThreads) == 0, "whole vectors per thread");
  Raw8<T> r[kIt];
  __device__ __forceinline__ void load(const T *src, int T_, int tid) {
#pragma unroll
    for (int it = 0; it < kIt; ++it) {
      const int e = 8 * (tid + kThreads * it);
      if (e / W < T_) r[it].load(src + e);
    }
  }
  template <typename F>
  __device__ __forceinline__ void store(float *dst, int P, int T_, int tid, F f) const {
#pragma unroll
    for (int it = 0; it < kIt; ++it) {
      const int e = 8 * (tid + kThreads * it), t = e / W, c = e - t * W;
      if (t < T_)
#pragma unroll
        for (int u = 0; u < 8; ++u) dst[t * P + c + u] = f(r[it][u]);
    }
  }
};

template <int TR, int TC>
__device__ __forceinline__ void zero(float (&acc)[TR][TC]) {
#pragma unroll
  for (int r = 0; r < TR; ++r)
#pragma unroll
    for (int c = 0; c < TC; ++c) acc[r][c] = 0.f;
}

// One call's pointers and sizes (device pointers; see BackwardProblem).
struct BwdArgs {
  const void *q, *k, *v;
  const float *dout, *S0, *z0, *dSN, *dzN;
  float *dq, *dk, *dv, *dS0, *dz0;
  float *Asc, *Bsc;  // [BH][nch * kT][kT]: pass 1's masked A and Bm of every chunk, for pass 2
  float *gnum;  // [BH][N][DV]: gnum of every token
  float *gden;  // [BH][N]: gden of every token
  // sums over the nsub parts of each segment (part f of segment s at s * nsub + f):
  float *segS;  // [BH][nseg * nsub][DK * DV + DK]: phi(K)^T V, colsum phi(K)
  float *segU;  // [BH][nseg * nsub][DK * DV + DK]: phi(Q)^T gnum, phi(Q)^T gden
  long N;
  int seg_chunks, nseg;
  int sub_chunks, nsub;  // a segment's parts for the sum phases: nsub runs of sub_chunks chunks
  float eps;
};

enum BwdPhase : int { kSegSums = 0, kPass1 = 1, kGradSums = 2, kPass2 = 3 };

template <typename Tin, int DK, int DV, int kPhase>
__global__ void __launch_bounds__(kThreads, 1) causal_backward_kernel(const __grid_constant__ BwdArgs arg) {
  const Tin *__restrict__ q = static_cast<const Tin *>(arg.q);
  const Tin *__restrict__ k = static_cast<const Tin *>(arg.k);
  const Tin *__restrict__ v = static_cast<const Tin *>(arg.v);
  const float *__restrict__ dout = arg.dout;
  float *__restrict__ dq = arg.dq;
  float *__restrict__ dk_g = arg.dk;
  float *__restrict__ dv_g = arg.dv;
  const long N = arg.N;
  const float eps = arg.eps;
  using L = BwdSmem<DK, DV>;
  constexpr int KP = L::KP, VP = L::VP, AP = L::AP;
  constexpr int RK = DK / 16, RV = DV / 16;  // register tile widths over features and values
  extern __shared__ float sm[];
  float *S = sm;              // [DK][VP] state (pass 1), U (pass 2)
  float *z = S + DK * VP;     // [DK]     normalizer (pass 1), u (pass 2)
  float *Qs = z + DK;         // [kT][KP] phi(q)
  float *Ks = Qs + kT * KP;   // [kT][KP] phi(k)
  float *Vs = Ks + kT * KP;   // [kT][VP] v
  float *Gs = Vs + kT * VP;   // [kT][DV] dO, then gnum
  float *A = Gs + kT * DV;    // [kT][AP] phi(q_t).phi(k_j), j <= t
  float *Bm = A + kT * AP;    // [kT][AP] v_j.gnum_t + gden_t, j <= t
  float *den = Bm + kT * AP;  // [kT]
  float *gd = den + kT;       // [kT] gden

  const long bh = blockIdx.y;
  // the sum phases run one CTA per part of a segment, the passes one per segment
  constexpr bool kSumPhase = kPhase == kSegSums || kPhase == kGradSums;
  const int seg = kSumPhase ? (int)blockIdx.x / arg.nsub : (int)blockIdx.x;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const long nch = (N + kT - 1) / kT;
  long c_begin = (long)seg * arg.seg_chunks, c_end = min(nch, c_begin + arg.seg_chunks);
  if (kSumPhase) {
    const long b = c_begin + (long)(blockIdx.x % arg.nsub) * arg.sub_chunks;
    c_end = min(c_end, b + arg.sub_chunks);
    c_begin = b;  // at or past c_end: an empty part, whose sum is zero
  }
  constexpr int kSum = DK * DV + DK;  // one segment sum: matrix then vector
  const long nparts = (long)arg.nseg * arg.nsub;
  const Tin *qh = q + bh * N * DK, *kh = k + bh * N * DK, *vh = v + bh * N * DV;
  const float *oh = dout + bh * N * DV;
  float *dqh = dq + bh * N * DK, *dkh = dk_g + bh * N * DK, *dvh = dv_g + bh * N * DV;
  float *gnum_h = arg.gnum + bh * N * DV, *gden_h = arg.gden + bh * N;
  float *Ah = arg.Asc + bh * nch * kT * kT, *Bh = arg.Bsc + bh * nch * kT * kT;  // row t0 + t: chunk t0's row t
  const auto phi_f = [](float x) { return phi(x); };
  const auto id_f = [](float x) { return x; };

  // operand accessors (row, column) of the products below
  auto aQ = [&](int t, int i) { return Qs[t * KP + i]; };
  auto bKt = [&](int i, int j) { return Ks[j * KP + i]; };
  auto bS = [&](int i, int c) { return S[i * VP + c]; };
  auto bSt = [&](int c, int i) { return S[i * VP + c]; };
  auto bV = [&](int j, int c) { return Vs[j * VP + c]; };
  auto bVt = [&](int c, int j) { return Vs[j * VP + c]; };
  auto aG = [&](int t, int c) { return Gs[t * DV + c]; };

  // starting state: pass 1 from S0 plus the earlier segments' sums; the sum phases from zero
  {
    const float *part = arg.segS + bh * nparts * kSum;
    for (int e = tid; e < DK * DV + DK; e += kThreads) {
      float x = 0.f;
      if (kPhase == kPass1) {
        x = e < DK * DV ? (arg.S0 ? arg.S0[bh * DK * DV + e] : 0.f) : (arg.z0 ? arg.z0[bh * DK + e - DK * DV] : 0.f);
        for (long s2 = 0; s2 < (long)seg * arg.nsub; ++s2) x += part[s2 * kSum + e];
      }
      if (e < DK * DV) S[(e / DV) * VP + e % DV] = x;
      else z[e - DK * DV] = x;
    }
  }

  // masked scores A = tril(phi(Q) phi(K)^T)
  auto scores = [&](int T) {
    float acc[4][4];
    zero(acc);
    tile_fma(acc, DK, ty, tx, aQ, bKt);
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int t = ty + 16 * r, j = tx + 16 * c;
        A[t * AP + j] = (j <= t && t < T) ? acc[r][c] : 0.f;
      }
  };

  if constexpr (kPhase == kSegSums) {
    // phi(K)^T V and colsum phi(K) over the segment
    for (long ci = c_begin; ci < c_end; ++ci) {
      const long t0 = ci * kT;
      const int T = (int)min((long)kT, N - t0);
      ChunkRows<DK, Tin> lk;
      ChunkRows<DV, Tin> lv;
      lk.load(kh + t0 * DK, T, tid);
      lv.load(vh + t0 * DV, T, tid);
      __syncthreads();  // the previous chunk is fully consumed
      lk.store(Ks, KP, T, tid, phi_f);
      lv.store(Vs, VP, T, tid, id_f);
      __syncthreads();
      float acc[RK][RV];
      zero(acc);
      tile_fma(acc, T, ty, tx, [&](int i, int j) { return Ks[j * KP + i]; }, bV);
#pragma unroll
      for (int r = 0; r < RK; ++r)
#pragma unroll
        for (int c = 0; c < RV; ++c) S[(ty + 16 * r) * VP + tx + 16 * c] += acc[r][c];
      for (int i = tid; i < DK; i += kThreads) {
        float sum = 0.f;
        for (int j = 0; j < T; ++j) sum += Ks[j * KP + i];
        z[i] += sum;
      }
    }
    __syncthreads();
    float *dst = arg.segS + (bh * nparts + blockIdx.x) * kSum;
    for (int e = tid; e < DK * DV + DK; e += kThreads) dst[e] = e < DK * DV ? S[(e / DV) * VP + e % DV] : z[e - DK * DV];
    return;
  }

  if constexpr (kPhase == kGradSums) {
    // phi(Q)^T gnum and phi(Q)^T gden over the segment (the first segment's is never read)
    if (seg == 0) return;
    for (long ci = c_begin; ci < c_end; ++ci) {
      const long t0 = ci * kT;
      const int T = (int)min((long)kT, N - t0);
      ChunkRows<DK, Tin> lq;
      ChunkRows<DV, float> lg;
      lq.load(qh + t0 * DK, T, tid);
      lg.load(gnum_h + t0 * DV, T, tid);
      const float gd_t = tid < T ? __ldg(gden_h + t0 + tid) : 0.f;  // kThreads >= kT
      __syncthreads();  // the previous chunk is fully consumed
      lq.store(Qs, KP, T, tid, phi_f);
      lg.store(Gs, DV, T, tid, id_f);
      if (tid < T) gd[tid] = gd_t;
      __syncthreads();
      float acc[RK][RV];
      zero(acc);
      tile_fma(acc, T, ty, tx, [&](int i, int t) { return Qs[t * KP + i]; }, [&](int t, int c) { return Gs[t * DV + c]; });
#pragma unroll
      for (int r = 0; r < RK; ++r)
#pragma unroll
        for (int c = 0; c < RV; ++c) S[(ty + 16 * r) * VP + tx + 16 * c] += acc[r][c];
      for (int i = tid; i < DK; i += kThreads) {
        float sum = 0.f;
        for (int t = 0; t < T; ++t) sum = fmaf(Qs[t * KP + i], gd[t], sum);
        z[i] += sum;
      }
    }
    __syncthreads();
    float *dst = arg.segU + (bh * nparts + blockIdx.x) * kSum;
    for (int e = tid; e < DK * DV + DK; e += kThreads) dst[e] = e < DK * DV ? S[(e / DV) * VP + e % DV] : z[e - DK * DV];
    return;
  }

  // ---------------- pass 1: chunks in order ----------------
  if constexpr (kPhase == kPass1) for (long t0 = c_begin * kT; t0 < c_end * kT && t0 < N; t0 += kT) {
    const int T = (int)min((long)kT, N - t0);
    ChunkRows<DK, Tin> lq, lk;
    ChunkRows<DV, Tin> lv;
    ChunkRows<DV, float> lo;
    lq.load(qh + t0 * DK, T, tid);
    lk.load(kh + t0 * DK, T, tid);
    lv.load(vh + t0 * DV, T, tid);
    lo.load(oh + t0 * DV, T, tid);
    __syncthreads();  // the previous chunk is fully consumed
    lq.store(Qs, KP, T, tid, phi_f);
    lk.store(Ks, KP, T, tid, phi_f);
    lv.store(Vs, VP, T, tid, id_f);
    lo.store(Gs, DV, T, tid, id_f);
    __syncthreads();
    scores(T);
    __syncthreads();
    {
      // four lanes per token, each a quarter of phi(q_t).z and of the row sum of A (rotated
      // start columns keep the 32 lanes of a warp on distinct banks)
      static_assert(kThreads == 4 * kT, "four lanes per token");
      const int t = tid >> 2, part = tid & 3;
      constexpr int QI = DK / 4;
      float d = 0.f, a = 0.f;
#pragma unroll 4
      for (int m = 0; m < QI; ++m) {
        const int i = part * QI + (m + 8 * part) % QI;
        d = fmaf(Qs[t * KP + i], z[i], d);
      }
#pragma unroll 4
      for (int m = 0; m < kT / 4; ++m) {
        const int j = part * (kT / 4) + m;
        if (j <= t) a += A[t * AP + j];
      }
      d += __shfl_xor_sync(0xffffffffu, d, 1);
      a += __shfl_xor_sync(0xffffffffu, a, 1);
      d += __shfl_xor_sync(0xffffffffu, d, 2);
      a += __shfl_xor_sync(0xffffffffu, a, 2);
      if (part == 0 && t < T) den[t] = (d + a) + eps;
    }
    // dO_t . o_t = (phi(q_t) . Y_t + sum_j A_tj C_tj) / den_t with Y = dO S_prev^T and C = dO V^T;
    // Y_t / den_t is also dq's state term, so one product serves both
    float accy[4][RK];  // Y, rows 4 ty .. 4 ty + 3
    {
      // C, masked (j <= t < T), in Bm's slot until Bm is formed from it
      float acc[4][4];
      zero(acc);
      tile_fma(acc, DV, ty, tx, aG, bVt);
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int t = ty + 16 * r, j = tx + 16 * c;
          Bm[t * AP + j] = (j <= t && t < T) ? acc[r][c] : 0.f;
        }
    }
    zero(accy);
    tile_fma<4, RK, true>(accy, 0, DV, ty, tx, aG, bSt);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      // phi(q_t) . Y_t, held in gd[t] until gden_t replaces it
      const int t = 4 * ty + r;
      float x = 0.f;
      if (t < T)
#pragma unroll
        for (int c = 0; c < RK; ++c) x = fmaf(Qs[t * KP + tx + 16 * c], accy[r][c], x);
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
      if (tx == 0 && t < T) gd[t] = x;
    }
    __syncthreads();
    {
      // gden_t = -(dO_t . o_t) / den_t, four lanes per token for sum_j A_tj C_tj
      const int t = tid >> 2, part = tid & 3;
      float ac = 0.f;
#pragma unroll 4
      for (int m = 0; m < kT / 4; ++m) {
        const int j = part * (kT / 4) + m;
        ac = fmaf(A[t * AP + j], Bm[t * AP + j], ac);
      }
      ac += __shfl_xor_sync(0xffffffffu, ac, 1);
      ac += __shfl_xor_sync(0xffffffffu, ac, 2);
      if (part == 0 && t < T) {
        const float dt = den[t];
        gd[t] = -((gd[t] + ac) / dt) / dt;
      }
    }
    __syncthreads();
    // gnum = dO / den; Bm = tril(C / den + gden), the masked score gradients
    for (int e = tid; e < T * DV; e += kThreads) Gs[e] /= den[e / DV];
    for (int e = tid; e < kT * kT; e += kThreads) {
      const int t = e / kT, j = e - t * kT;
      Bm[t * AP + j] = (j <= t && t < T) ? Bm[t * AP + j] / den[t] + gd[t] : 0.f;
    }
    __syncthreads();
    for (int e = tid; e < T * DV; e += kThreads) gnum_h[t0 * DV + e] = Gs[e];
    for (int t = tid; t < T; t += kThreads) gden_h[t0 + t] = gd[t];
    // A and Bm for pass 2, which reads them instead of forming them again
    for (int e = tid; e < kT * kT; e += kThreads) {
      const int t = e / kT, j = e - t * kT;
      Ah[t0 * kT + e] = A[t * AP + j];
      Bh[t0 * kT + e] = Bm[t * AP + j];
    }
    {
      // dphi(q_t) = Y_t / den_t + z_prev gden_t + sum_{j <= t} Bm_tj phi(k_j)
      // rows 4 ty .. 4 ty + 3: Bm_tj is zero past j = t
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int t = 4 * ty + r;
        if (t < T)
#pragma unroll
          for (int c = 0; c < RK; ++c) accy[r][c] /= den[t];
      }
      tile_fma<4, RK, true>(accy, 0, min(T, 4 * ty + 4), ty, tx, [&](int t, int j) { return Bm[t * AP + j]; },
                            [&](int j, int i) { return Ks[j * KP + i]; });
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int t = 4 * ty + r;
        if (t < T)
#pragma unroll
          for (int c = 0; c < RK; ++c) {
            const int i = tx + 16 * c;
            dqh[(t0 + t) * DK + i] = (accy[r][c] + z[i] * gd[t]) * fminf(Qs[t * KP + i], 1.f);
          }
      }
    }
    __syncthreads();
    {
      // fold the chunk into the state: S += phi(K)^T V, z += colsum phi(K)
      float acc[RK][RV];
      zero(acc);
      tile_fma(acc, T, ty, tx, [&](int i, int j) { return Ks[j * KP + i]; }, bV);
#pragma unroll
      for (int r = 0; r < RK; ++r)
#pragma unroll
        for (int c = 0; c < RV; ++c) S[(ty + 16 * r) * VP + tx + 16 * c] += acc[r][c];
      for (int i = tid; i < DK; i += kThreads) {
        float s = 0.f;
        for (int j = 0; j < T; ++j) s += Ks[j * KP + i];
        z[i] += s;
      }
    }
  }

  if constexpr (kPhase == kPass1) return;

  // ---------------- pass 2: chunks in reverse ----------------
  // U, u at the segment's end: dS, dz plus the later segments' gradient sums
  {
    const float *part = arg.segU + bh * nparts * kSum;
    __syncthreads();
    for (int e = tid; e < DK * DV + DK; e += kThreads) {
      float x = e < DK * DV ? (arg.dSN ? arg.dSN[bh * DK * DV + e] : 0.f)
                            : (arg.dzN ? arg.dzN[bh * DK + e - DK * DV] : 0.f);
      for (long s2 = (long)(seg + 1) * arg.nsub; s2 < nparts; ++s2) x += part[s2 * kSum + e];
      if (e < DK * DV) S[(e / DV) * VP + e % DV] = x;
      else z[e - DK * DV] = x;
    }
  }
  for (long ci = c_end - 1; ci >= c_begin; --ci) {
    const long t0 = ci * kT;
    const int T = (int)min((long)kT, N - t0);
    ChunkRows<DK, Tin> lq, lk;
    ChunkRows<DV, Tin> lv;
    ChunkRows<DV, float> lg;
    lq.load(qh + t0 * DK, T, tid);
    lk.load(kh + t0 * DK, T, tid);
    lv.load(vh + t0 * DV, T, tid);
    lg.load(gnum_h + t0 * DV, T, tid);
    const float gd_t = tid < T ? __ldg(gden_h + t0 + tid) : 0.f;  // kThreads >= kT
    ChunkRows<kT, float> la, lb;  // pass 1's A and Bm (all kT rows: zero past T)
    la.load(Ah + t0 * kT, kT, tid);
    lb.load(Bh + t0 * kT, kT, tid);
    __syncthreads();  // the previous chunk is fully consumed
    lq.store(Qs, KP, T, tid, phi_f);
    lk.store(Ks, KP, T, tid, phi_f);
    lv.store(Vs, VP, T, tid, id_f);
    lg.store(Gs, DV, T, tid, id_f);
    la.store(A, AP, kT, tid, id_f);
    lb.store(Bm, AP, kT, tid, id_f);
    if (tid < T) gd[tid] = gd_t;
    __syncthreads();
    {
      // dphi(k_j) = U v_j + u + sum_{t >= j} Bm_tj phi(q_t)
      // rows 4 ty .. 4 ty + 3: Bm_tj is zero before t = j
      float acc[4][RK];
      zero(acc);
      tile_fma<4, RK, true>(acc, 0, DV, ty, tx, [&](int j, int c) { return Vs[j * VP + c]; }, bSt);
      tile_fma<4, RK, true>(acc, 4 * ty, T, ty, tx, [&](int j, int t) { return Bm[t * AP + j]; },
                            [&](int t, int i) { return Qs[t * KP + i]; });
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int j = 4 * ty + r;
        if (j < T)
#pragma unroll
          for (int c = 0; c < RK; ++c) {
            const int i = tx + 16 * c;
            dkh[(t0 + j) * DK + i] = (acc[r][c] + z[i]) * fminf(Ks[j * KP + i], 1.f);
          }
      }
    }
    {
      // dv_j = U^T phi(k_j) + sum_{t >= j} A_tj gnum_t
      // rows 4 ty .. 4 ty + 3: A_tj is zero before t = j
      float acc[4][RV];
      zero(acc);
      tile_fma<4, RV, true>(acc, 0, DK, ty, tx, [&](int j, int i) { return Ks[j * KP + i]; }, bS);
      tile_fma<4, RV, true>(acc, 4 * ty, T, ty, tx, [&](int j, int t) { return A[t * AP + j]; },
                            [&](int t, int c) { return Gs[t * DV + c]; });
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int j = 4 * ty + r;
        if (j < T)
#pragma unroll
          for (int c = 0; c < RV; ++c) dvh[(t0 + j) * DV + tx + 16 * c] = acc[r][c];
      }
    }
    __syncthreads();
    {
      // U += phi(Q)^T gnum, u += phi(Q)^T gden
      float acc[RK][RV];
      zero(acc);
      tile_fma(acc, T, ty, tx, [&](int i, int t) { return Qs[t * KP + i]; }, [&](int t, int c) { return Gs[t * DV + c]; });
#pragma unroll
      for (int r = 0; r < RK; ++r)
#pragma unroll
        for (int c = 0; c < RV; ++c) S[(ty + 16 * r) * VP + tx + 16 * c] += acc[r][c];
      for (int i = tid; i < DK; i += kThreads) {
        float s = 0.f;
        for (int t = 0; t < T; ++t) s = fmaf(Qs[t * KP + i], gd[t], s);
        z[i] += s;
      }
    }
  }
  __syncthreads();
  if (seg == 0 && arg.dS0)
    for (int e = tid; e < DK * DV; e += kThreads) arg.dS0[bh * DK * DV + e] = S[(e / DV) * VP + e % DV];
  if (seg == 0 && arg.dz0)
    for (int i = tid; i < DK; i += kThreads) arg.dz0[bh * DK + i] = z[i];
}

template <typename Tin, int DK, int DV, int kPhase>
cudaError_t launch_phase(const BwdArgs &a, dim3 grid, cudaStream_t stream) {
  constexpr size_t smem = BwdSmem<DK, DV>::Bytes;
  cudaError_t e = cudaFuncSetAttribute(causal_backward_kernel<Tin, DK, DV, kPhase>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  causal_backward_kernel<Tin, DK, DV, kPhase><<<grid, kThreads, smem, stream>>>(a);
  e = cudaGetLastError();
  if (e == cudaSuccess) count_launch();
  return e;
}

template <typename Tin, int DK, int DV>
cudaError_t launch_t(const BwdArgs &a, int BH, cudaStream_t stream) {
  LaunchTimer timer(kKBackward, stream);
  cudaError_t e = cudaSuccess;
  if (a.nseg > 1) e = launch_phase<Tin, DK, DV, kSegSums>(a, dim3((a.nseg - 1) * a.nsub, BH), stream);
  if (e == cudaSuccess) e = launch_phase<Tin, DK, DV, kPass1>(a, dim3(a.nseg, BH), stream);
  if (e == cudaSuccess && a.nseg > 1) e = launch_phase<Tin, DK, DV, kGradSums>(a, dim3(a.nseg * a.nsub, BH), stream);
  if (e == cudaSuccess) e = launch_phase<Tin, DK, DV, kPass2>(a, dim3(a.nseg, BH), stream);
  timer.done(e);
  return e;
}

template <typename Tin, int DK>
cudaError_t launch_dv(const BwdArgs &a, int BH, int dv, cudaStream_t s) {
  if (dv == 32) return launch_t<Tin, DK, 32>(a, BH, s);
  if (dv == 64) return launch_t<Tin, DK, 64>(a, BH, s);
  return launch_t<Tin, DK, 128>(a, BH, s);
}

template <typename Tin>
cudaError_t launch_dk(const BwdArgs &a, int BH, int dk, int dv, cudaStream_t s) {
  if (dk == 32) return launch_dv<Tin, 32>(a, BH, dv, s);
  if (dk == 64) return launch_dv<Tin, 64>(a, BH, dv, s);
  return launch_dv<Tin, 128>(a, BH, dv, s);
}

}  // namespace

cudaError_t launch_causal_backward(const BackwardProblem &b) {
  const Problem &p = b.p;
  // segments per head: enough CTAs to cover the SMs once, at least 4 chunks each
  const long nch = (p.N + kT - 1) / kT;
  const long sms = std::max(1, device_info(-1).sm_count);
  long nseg = std::max(1L, std::min(sms / std::max(1, p.BH), nch / 4));
  const long seg_chunks = std::max(1L, (nch + nseg - 1) / nseg);
  nseg = std::max(1L, (nch + seg_chunks - 1) / seg_chunks);
  // the sum phases cut each segment into nsub parts, so that their CTAs (B H (nseg - 1) nsub
  // with work) also cover the SMs about once
  long nsub = 1;
  if (nseg > 1) nsub = std::max(1L, std::min(seg_chunks, sms / std::max(1L, (long)p.BH * (nseg - 1))));
  const long sub_chunks = (seg_chunks + nsub - 1) / nsub;
  nsub = (seg_chunks + sub_chunks - 1) / sub_chunks;
  // scratch: A and Bm of every chunk, gnum and gden of every token, then the part sums of the
  // state and of the gradients; each block starts on a 256-byte boundary (g_f is rounded up
  // to 64 floats, and every other block size is a multiple of 32 floats)
  const size_t sum_f = (size_t)p.dk * p.dv + p.dk;
  const size_t ab_f = (size_t)p.BH * nch * kT * kT;
  // (with one segment no part sums exist, and the passes read none)
  const size_t g_f = (2 * ab_f + (size_t)p.BH * p.N * (p.dv + 1) + 63) / 64 * 64;
  const size_t seg_f = nseg > 1 ? (size_t)p.BH * nseg * nsub * sum_f : 0;
  float *G = nullptr;
  cudaError_t e = cudaMallocAsync(reinterpret_cast<void **>(&G), std::max<size_t>(sizeof(float) * (g_f + 2 * seg_f), 16),
                                  p.stream);
  if (e != cudaSuccess) return e;
  BwdArgs a;
  a.q = p.q, a.k = p.k, a.v = p.v;
  a.dout = b.dout, a.S0 = b.S0, a.z0 = b.z0, a.dSN = b.dS, a.dzN = b.dz;
  a.dq = b.dq, a.dk = b.dk, a.dv = b.dv, a.dS0 = b.dS0, a.dz0 = b.dz0;
  a.Asc = G, a.Bsc = G + ab_f;
  a.gnum = G + 2 * ab_f, a.gden = a.gnum + (size_t)p.BH * p.N * p.dv, a.segS = G + g_f, a.segU = G + g_f + seg_f;
  a.N = p.N, a.seg_chunks = (int)seg_chunks, a.nseg = (int)nseg, a.eps = p.eps;
  a.sub_chunks = (int)sub_chunks, a.nsub = (int)nsub;
  e = p.dt == LA_F32 ? launch_dk<float>(a, p.BH, p.dk, p.dv, p.stream)
                     : launch_dk<__nv_bfloat16>(a, p.BH, p.dk, p.dv, p.stream);
  const cudaError_t f = cudaFreeAsync(G, p.stream);
  return e != cudaSuccess ? e : f;
}

}  // namespace la
