// Gradient of the causal prefill on the sm_103a tensor cores (tcgen05, TMEM).
//
// The forward is o_t = phi(q_t)^T S_t / (phi(q_t)^T z_t + eps) with the state
// inclusive of token t ("线性注意力从头到尾讲清楚" §7; "Linear Attention Math",
// "The recurrent form").  The pages name training through chunked matrix
// products ("Linear Attention: From Pairwise Reads to a Recurrent State", "A
// recurrence need not force token-serial training"; "Linear in which
// variable?": chunk boundary states and gradients) but write no backward
// pass; this is the derivative of the definition, in 128-token chunks.
// Within a chunk (rows t = queries, j = keys, i = key features, c = value
// components), with Q = phi(q), K = phi(k) and the state S_prev, z_prev
// carried in from the earlier chunks:
//   A    = tril(Q K^T),  C = tril(dO V^T),  Y = dO S_prev^T
//   den  = Q z_prev + rowsum(A) + eps
//   gden = -(rowsum(Q * Y) + rowsum(A * C)) / den^2          (= -(dO . o) / den)
//   B'   = tril(C + den gden)                                (= den * dO-score gradient)
//   dQ   = ((Y + B' K) / den + gden z_prev^T) * phi'(q)
// and in reverse order, with U, u the gradient of the state carried in from
// the later chunks (dS, dz at the end) and gnum = dO / den:
//   dV   = K U + triu(K Q^T) gnum
//   dK   = (V U^T + triu(V gnum^T + gden) Q + u) * phi'(k)
//   U   += Q^T gnum,  u += Q^T gden.
// phi = ELU + 1 gives phi'(x) = min(phi(x), 1).
//
// Precision.  At early tokens the query gradient is a difference of terms
// about a thousand times larger than itself, so every operand that is not a
// bf16 input (Q, K, dO, S_prev, B', U, the key-side scores and gnum) reaches
// the tensor cores as a bf16 pair hi + lo (hi = bf16(x), lo = bf16(x - hi),
// about 16 significant bits); a product of two pairs is taken as
// hi hi + hi lo + lo hi, a pair against V as two products.  All
// accumulation is fp32 in tensor memory; den, gden, z and u are fp32.
//
// Two kernels, one CTA per head (a CTA carries its head's state through all
// chunks in order):
//   pass 1 (chunks in order): dq, and den, gden of every token for pass 2;
//   pass 2 (chunks in reverse), two CTA roles per head: role 0 computes dv
//     and the initial state's dS0, role 1 dk and dz0; both carry U.
// Operands are staged by threads from global memory (one chunk ahead in L2
// through bulk prefetches) into 128-byte-swizzled shared tiles or straight
// into tensor memory; one thread issues the MMAs.  Every mbarrier wait is
// bounded: a wait that runs out raises the CTA's abort word and the device
// status word, the CTA drains its MMAs, frees tensor memory and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace la {

__device__ unsigned int g_bwd_status;

namespace {
using namespace tc;

constexpr int kC = 128;               // tokens per chunk
constexpr int kD = 128;               // d_k = d_v
constexpr uint32_t kBlk = 16384;      // [128 rows x 64] bf16, 128-byte swizzled
constexpr uint32_t kTile = 2 * kBlk;  // [128 x 128] bf16 tile
constexpr uint32_t kAbortMisaligned = 2u;

// ---------------------------------------------------------------------------
// Small helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float lo16(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi16(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
// phi(a), phi(b) in fp32: x + 1 above zero, e^x = 2^(x log2 e) on the MUFU unit
// below (relative error near 2^-22, far below the 2^-17 of a bf16 pair).
__device__ __forceinline__ float2 phi2(float a, float b) {
  const float2 y = __fmul2_rn(make_float2(a, b), make_float2(1.4426950408889634f, 1.4426950408889634f));
  return make_float2(a > 0.f ? a + 1.f : ex2_approx(y.x), b > 0.f ? b + 1.f : ex2_approx(y.y));
}

// Two fp32 values as a bf16 pair: hi word (a, b), lo word (a - hi_a, b - hi_b).
__device__ __forceinline__ void split2(float a, float b, uint32_t &h, uint32_t &l) {
  h = pack_bf16(a, b);
  l = pack_bf16(a - lo16(h), b - hi16(h));
}

// phi of the eight bf16 inputs packed in x, as bf16 pairs (hi, lo words of
// feature pairs); v receives hi + lo, the values the tensor cores see.
__device__ __forceinline__ void phi_split8(uint4 x, uint32_t (&h)[4], uint32_t (&l)[4], float (&v)[8]) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 f = phi2(lo16(w[e]), hi16(w[e]));
    split2(f.x, f.y, h[e], l[e]);
    v[2 * e] = lo16(h[e]) + lo16(l[e]);
    v[2 * e + 1] = hi16(h[e]) + hi16(l[e]);
  }
}

// As phi_split8 without the values: the pair words of eight phi values.
__device__ __forceinline__ void phi_pair8(uint4 x, uint4 &h, uint4 &l) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
  uint32_t hh[4], ll[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 f = phi2(lo16(w[e]), hi16(w[e]));
    split2(f.x, f.y, hh[e], ll[e]);
  }
  h = make_uint4(hh[0], hh[1], hh[2], hh[3]);
  l = make_uint4(ll[0], ll[1], ll[2], ll[3]);
}

// 32-byte global load (read-only path) and store; the address must be 32-byte aligned.
__device__ __forceinline__ void ld_row32(const void *p, uint32_t (&r)[8]) {
  asm volatile("ld.global.nc.v8.u32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "l"(p));
}
__device__ __forceinline__ void st_row32(void *p, const uint32_t *r) {
  asm volatile("st.global.v8.u32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(r[0]), "r"(r[1]), "r"(r[2]),
               "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}

// K-major operand over a [128 x 128] tile (rows of 64 K-elements per block).
__device__ __forceinline__ uint64_t kdesc(uint32_t tile, int ks) {
  return sw128_desc(tile + (ks >> 2) * kBlk + (ks & 3) * 32, 16, 1024);
}
// MN-major operand over a [128 x 128] tile (rows = K index, two 64-wide blocks).
__device__ __forceinline__ uint64_t mndesc(uint32_t tile, int ks) {
  return sw128_desc(tile + ks * 2048, kBlk, 1024);
}

// Row `row`, columns col0 .. col0 + 7 of a [128 x 128] bf16 tile.
__device__ __forceinline__ uint4 *tile_chunk(uint8_t *tile, int row, int col0) {
  return reinterpret_cast<uint4 *>(tile + (col0 >> 6) * kBlk + sw128_offset(row, col0 & 63));
}

// Split 32 fp32 score columns (keys 32 cb .. 32 cb + 31 of this lane's row) in
// place into bf16 pairs for use as a tensor-memory A operand: every 16 keys
// become 8 columns of hi pairs then 8 of lo pairs.  keep(j) selects the
// entries kept (the others become zeros); f(j, x) transforms a kept value.
template <typename Keep, typename F>
__device__ __forceinline__ void split_scores32(uint32_t (&r)[32], int cb, Keep keep, F f) {
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    uint32_t o[16];
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const int j = cb * 32 + g * 16 + 2 * m;
      const float a = keep(j) ? f(j, __uint_as_float(r[g * 16 + 2 * m])) : 0.f;
      const float b = keep(j + 1) ? f(j + 1, __uint_as_float(r[g * 16 + 2 * m + 1])) : 0.f;
      split2(a, b, o[m], o[8 + m]);
    }
#pragma unroll
    for (int e = 0; e < 16; ++e) r[g * 16 + e] = o[e];
  }
}

// Arguments of both passes (device pointers; [BH][N][128] rows, fp32 unless noted).
struct BwdTcParams {
  CUtensorMap tq, tk, tv;  // [BH][N][128] bf16, boxes of 64 features x 128 tokens, 128-byte swizzle
  const __nv_bfloat16 *q, *k, *v;  // inputs
  const float *dout;
  const float *S0, *z0;  // initial state (nullable)
  const float *dS, *dz;  // gradient of the final state (nullable)
  float *dq, *dk, *dv;
  float *dS0, *dz0;  // gradient of the initial state (nullable)
  float *den, *gden;  // [BH][N]: written by pass 1, read by pass 2
  // pass 1's segment split: nseg segments of seg_chunks chunks per head; the state pass sums
  // segment s < nseg - 1 in `parts` pieces, piece (bh, s, f) at part_S[((bh (nseg - 1) + s) parts
  // + f) 128 x 128] and part_z[... 128]
  float *part_S, *part_z;
  int seg_chunks, nseg, parts;
  long N;
  float eps;
};

// Features 64 h .. 64 h + 63 of a 128-element bf16 row, by four 32-byte loads.
__device__ __forceinline__ void load_row_half(const __nv_bfloat16 *row, uint4 (&x)[8], int h = 0) {
  const uint8_t *src = reinterpret_cast<const uint8_t *>(row) + 128 * h;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    uint32_t w[8];
    ld_row32(src + 32 * e, w);
    x[2 * e] = make_uint4(w[0], w[1], w[2], w[3]);
    x[2 * e + 1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

// phi pairs of features 64 h .. 64 h + 63 of this lane's query row into the
// tensor-memory phi(Q) columns (hi at kP1Q + 32 h .., lo at kP1Q + 64 + 32 h ..;
// zeros for an invalid row); returns their part of phi(q) . z.
__device__ __forceinline__ float query_pairs_half(const uint4 (&x)[8], bool valid, const float *z, uint32_t tl, int h);

// phi pairs of a raw [128 x 128] bf16 tile in place: hi over the raw values,
// lo into the matching chunks of `lo`.  Thread u (of 256) takes the 16-byte
// chunks u + 256 i; chunk ch is row (ch mod 1024) / 8 of block ch / 1024 and
// rows past the T valid ones become zeros.
__device__ __forceinline__ void key_pairs(uint4 *hi, uint4 *lo, int u, int T) {
#pragma unroll 4
  for (int i = 0; i < 8; ++i) {
    const int ch = u + 256 * i;
    uint4 h = make_uint4(0u, 0u, 0u, 0u), l = h;
    if (((ch & 1023) >> 3) < T) phi_pair8(hi[ch], h, l);
    hi[ch] = h;
    lo[ch] = l;
  }
}

// Column sums of the valid rows of a pair of [128 x 128] bf16 tiles (hi + lo)
// over 128 threads: thread g takes the column pair 2 p, 2 p + 1 with
// p = (g & 15) + 16 (g >> 5) over rows of one half ((g >> 4) & 1); the halves
// meet through a shuffle and lanes 0-15 of each warp hold the pair's sums.
__device__ __forceinline__ float2 pair_column_sums(const uint8_t *hi, const uint8_t *lo, int g, int T) {
  const int p = (g & 15) + 16 * (g >> 5), half = (g >> 4) & 1;
  const int col = 2 * p;
  const uint32_t boff = (col >> 6) * kBlk;
  float2 s = make_float2(0.f, 0.f);
  const int r0 = 64 * half, r1 = min(T, r0 + 64);
#pragma unroll 8
  for (int j = r0; j < r1; ++j) {
    const uint32_t off = boff + sw128_offset(j, col & 63);
    const uint32_t a = *reinterpret_cast<const uint32_t *>(hi + off), b = *reinterpret_cast<const uint32_t *>(lo + off);
    s = __fadd2_rn(s, __fadd2_rn(make_float2(lo16(a), hi16(a)), make_float2(lo16(b), hi16(b))));
  }
  s.x += __shfl_xor_sync(0xffffffffu, s.x, 16);
  s.y += __shfl_xor_sync(0xffffffffu, s.y, 16);
  return s;
}

// ---------------------------------------------------------------------------
// State pass for pass 1's segment split: the sums phi(K)^T V and colsum phi(K)
// over parts of the earlier segments, with phi(K) as bf16 pairs (the same
// operands and fp32 accumulation as pass 1's own state update).
// ---------------------------------------------------------------------------
struct StLayout {
  static constexpr int kStages = 2;
  static constexpr uint32_t K = 0;                       // raw keys, then the hi pairs in place
  static constexpr uint32_t Klo = kStages * kTile;       // lo pairs
  static constexpr uint32_t V = 2 * kStages * kTile;
  static constexpr uint32_t Bars = 3 * kStages * kTile;  // full, phi_done, empty per stage; acc_full, drain
  static constexpr uint32_t Misc = Bars + (3 * kStages + 2) * 8;
  static constexpr uint32_t Bytes = Misc + 16;
};
static_assert(StLayout::Bytes <= 232448, "state pass shared memory");
constexpr int kStThreads = 320;  // warp 0 TMA, 1 MMA, 2-9 phi pairs (2-5 also key column sums and the output)
constexpr uint32_t kBarSt = 1;

__global__ void __launch_bounds__(kStThreads, 1) bwd_state_tc(const __grid_constant__ BwdTcParams p) {
  using L = StLayout;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) atomicOr(&g_bwd_status, kAbortMisaligned);
    return;
  }
  uint8_t *sm = smem_raw;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::Bars);
  uint64_t *full = bars, *phi_done = bars + L::kStages, *empty = bars + 2 * L::kStages,
           *acc_full = bars + 3 * L::kStages, *drain = acc_full + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + L::Misc);
  volatile uint32_t *abort_word = reinterpret_cast<volatile uint32_t *>(sm + L::Misc + 4);
  unsigned int *status = &g_bwd_status;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.y;
  const int sgm = blockIdx.x / p.parts, part = blockIdx.x % p.parts;  // segment sgm < nseg - 1
  const long N = p.N;
  const int nch = (int)((N + kC - 1) / kC);
  // this part's chunks [cb, ce) of segment sgm
  const int s0 = sgm * p.seg_chunks, s1 = min(nch, s0 + p.seg_chunks);
  const int cb = s0 + (int)((long)(s1 - s0) * part / p.parts), ce = s0 + (int)((long)(s1 - s0) * (part + 1) / p.parts);
  const int n = max(0, ce - cb);
  if (threadIdx.x == 0) {
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&phi_done[s], 256);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(drain, 1);
    *abort_word = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, 128);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const long piece = ((long)bh * (p.nseg - 1) + sgm) * p.parts + part;

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&p.tk);
      prefetch_tmap(&p.tv);
      int issued = 0;
      for (int i = 0; i < n; ++i) {
        const int s = i % L::kStages;
        if (i >= L::kStages && !mbar_wait(&empty[s], ((i / L::kStages) - 1) & 1, abort_word, status)) break;
        const int tok = (cb + i) * kC;
        mbar_arrive_expect_tx(&full[s], 2 * kTile);
        tma_load_3d(sm + L::K + s * kTile, &p.tk, &full[s], 0, tok, bh);
        tma_load_3d(sm + L::K + s * kTile + kBlk, &p.tk, &full[s], 64, tok, bh);
        tma_load_3d(sm + L::V + s * kTile, &p.tv, &full[s], 0, tok, bh);
        tma_load_3d(sm + L::V + s * kTile + kBlk, &p.tv, &full[s], 64, tok, bh);
        issued = i + 1;
      }
      for (int i = max(0, issued - L::kStages); i < issued; ++i)
        wait_drain(&full[i % L::kStages], (i / L::kStages) & 1, status);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t iMM = idesc_bf16_f32(128, 128, 1, 1);
      for (int i = 0; i < n; ++i) {
        const int s = i % L::kStages;
        if (!mbar_wait(&phi_done[s], (i / L::kStages) & 1, abort_word, status)) break;
        tc_fence_after();
        const uint32_t kh_ = smem_u32(sm + L::K + s * kTile), kl_ = smem_u32(sm + L::Klo + s * kTile),
                       v_ = smem_u32(sm + L::V + s * kTile);
#pragma unroll 4
        for (int ks = 0; ks < 8; ++ks) {
          mma_bf16(tmem, mndesc(kh_, ks), mndesc(v_, ks), iMM, (i > 0 || ks > 0) ? 1u : 0u);
          mma_bf16(tmem, mndesc(kl_, ks), mndesc(v_, ks), iMM, 1u);
        }
        mma_commit(&empty[s]);
      }
      mma_commit(acc_full);
      mma_commit(drain);
      wait_drain(drain, 0, status);
    }
  } else {
    // phi pairs in place over all 256 threads; threads 0-127 also sum the key columns
    const int g = threadIdx.x - 64;  // 0..255
    float2 zacc = make_float2(0.f, 0.f);
    bool ok = true;
    for (int i = 0; i < n; ++i) {
      const int s = i % L::kStages;
      const int T = (int)min((long)kC, N - (long)(cb + i) * kC);
      ok = mbar_wait(&full[s], (i / L::kStages) & 1, abort_word, status);
      if (bar_or(kBarSt, 256, !ok)) break;
      uint8_t *kt = sm + L::K + s * kTile, *lt = sm + L::Klo + s * kTile;
      key_pairs(reinterpret_cast<uint4 *>(kt), reinterpret_cast<uint4 *>(lt), g, T);
      named_bar(kBarSt, 256);
      if (g < 128) {
        const float2 cs = pair_column_sums(kt, lt, g, T);
        zacc.x += cs.x;
        zacc.y += cs.y;
      }
      fence_async_smem();
      mbar_arrive(&phi_done[s]);
    }
    // the piece: TMEM rows (features) to part_S, the key sums to part_z (threads 0-127)
    if (g < 128) {
      const int quarter = warp & 3, r = quarter * 32 + lane;
      ok = ok && (n == 0 || mbar_wait(acc_full, 0, abort_word, status));
      float *dst = p.part_S + (piece * kD + r) * kD;
      if (ok && n > 0) {
        tc_fence_after();
        const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
        for (int cb2 = 0; cb2 < 4; ++cb2) {
          uint32_t w[32];
          tmem_ld32(tl + cb2 * 32, w);
          float4 *d4 = reinterpret_cast<float4 *>(dst + cb2 * 32);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            d4[e] = make_float4(__uint_as_float(w[4 * e]), __uint_as_float(w[4 * e + 1]), __uint_as_float(w[4 * e + 2]),
                                __uint_as_float(w[4 * e + 3]));
        }
      } else if (n == 0) {
        for (int c = 0; c < kD; c += 4) *reinterpret_cast<float4 *>(dst + c) = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      if ((g & 31) < 16) {
        const int pc = 2 * ((g & 15) + 16 * (g >> 5));
        p.part_z[piece * kD + pc] = zacc.x;
        p.part_z[piece * kD + pc + 1] = zacc.y;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

// Shared-memory layout of pass 1: seven [128 x 128] bf16 tiles (224 KB), then
// two z buffers, the chunk's phi(q).z, barriers.
struct P1Layout {
  static constexpr uint32_t Khi = 0, Klo = kTile, V = 2 * kTile, Ghi = 3 * kTile, Glo = 4 * kTile, Shi = 5 * kTile,
                            Slo = 6 * kTile;
  static constexpr uint32_t Z = 7 * kTile;    // [2][128] z carried into the chunk
  static constexpr uint32_t DenX = Z + 1024;     // [2][128] phi(q_t) . z_prev over features 0-63, 64-127
  static constexpr uint32_t Kcol = DenX + 1024;  // [128] column sums of the chunk's phi(K)
  static constexpr uint32_t Bars = Kcol + 512;
  static constexpr int kNumBars = 18;
  static constexpr uint32_t Misc = Bars + kNumBars * 8;
  static constexpr uint32_t Bytes = Misc + 16;
};
static_assert(P1Layout::Bytes <= 232448, "pass 1 shared memory");

// TMEM columns of pass 1: S accumulator; two score regions that trade roles by
// chunk parity, so that the next chunk's A = Q K^T can go in while the dq phase
// still reads this chunk's Y + B' K: region RA(c) holds A, then Y and Y + B' K,
// region RC(c) holds C, then B' as bf16 pairs, and RA(c + 1) = RC(c); phi(Q)
// as bf16 pairs (hi 64 columns, lo 64).
constexpr uint32_t kP1S = 0, kP1X = 128, kP1CB = 256, kP1Q = 384;
__device__ __forceinline__ uint32_t p1_ra(int c) { return (c & 1) ? kP1CB : kP1X; }
__device__ __forceinline__ uint32_t p1_rc(int c) { return (c & 1) ? kP1X : kP1CB; }

// Warp roles of pass 1 (13 warps): 0 MMA issuer, tensor-memory owner and the
// key loads of chunks after the first (TMA); 1-4 half of the key pairs in
// place, queries 0-63 (phi pairs into tensor memory, one chunk ahead) and
// copies of the state; 5-8 dO pairs (and V by TMA, one chunk ahead), the other
// half of the key pairs, key column sums, queries 64-127; 9-12 scores, the
// next chunk's z, and dq.
constexpr int kP1Threads = 416;
constexpr int kP1WarpG = 5, kP1WarpE = 9;
constexpr uint32_t kBarQK = 1, kBarG = 2, kBarE = 3;

__device__ __forceinline__ float query_pairs_half(const uint4 (&x)[8], bool valid, const float *z, uint32_t tl, int h) {
  float dot = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    uint32_t hw[4] = {0u, 0u, 0u, 0u}, lw[4] = {0u, 0u, 0u, 0u};
    float vv[8];
    if (valid) {
      phi_split8(x[e], hw, lw, vv);
#pragma unroll
      for (int m = 0; m < 8; ++m) dot = fmaf(vv[m], z[64 * h + 8 * e + m], dot);
    }
    // features 64 h + 8 e .. + 7: pair columns 32 h + 4 e .. + 3 (hi), 64 + 32 h + 4 e .. (lo)
    tmem_st4_nowait(tl + kP1Q + 32 * h + 4 * e, hw[0], hw[1], hw[2], hw[3]);
    tmem_st4_nowait(tl + kP1Q + 64 + 32 * h + 4 * e, lw[0], lw[1], lw[2], lw[3]);
  }
  tmem_wait_st();
  return dot;
}

__global__ void __launch_bounds__(kP1Threads, 1) bwd_pass1_tc(const __grid_constant__ BwdTcParams p) {
  using L = P1Layout;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) atomicOr(&g_bwd_status, kAbortMisaligned);
    return;
  }
  uint8_t *sm = smem_raw;
  float *zbuf = reinterpret_cast<float *>(sm + L::Z);
  float *den_x = reinterpret_cast<float *>(sm + L::DenX);
  float *kcol = reinterpret_cast<float *>(sm + L::Kcol);
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::Bars);
  uint64_t *q_ready = bars + 0, *k_ready = bars + 1, *g_ready = bars + 2, *s_ready = bars + 3, *ac_full = bars + 4,
           *x_free = bars + 5, *y_full = bars + 6, *cb_ready = bars + 7, *d_full = bars + 8, *e3_done = bars + 9,
           *drain = bars + 10, *z_full = bars + 11 /* [2] */, *z_empty = bars + 13 /* [2] */, *k_full = bars + 15,
           *v_full = bars + 16, *kc_ready = bars + 17;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + L::Misc);
  volatile uint32_t *abort_word = reinterpret_cast<volatile uint32_t *>(sm + L::Misc + 4);
  unsigned int *status = &g_bwd_status;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // one CTA per (segment, head); the segment's chunks [c0, c0 + nloc) in order
  const int bh = blockIdx.y, seg = blockIdx.x;
  const long N = p.N;
  const int nch = (int)((N + kC - 1) / kC);
  const int c0 = seg * p.seg_chunks;
  const int nloc = min(nch, c0 + p.seg_chunks) - c0;
  const __nv_bfloat16 *qh = p.q + (long)bh * N * kD, *kh = p.k + (long)bh * N * kD, *vh = p.v + (long)bh * N * kD;
  const float *gh = p.dout + (long)bh * N * kD;

  if (threadIdx.x == 0) {
    mbar_init(q_ready, 256);  // both halves of the query pairs
    mbar_init(k_ready, 256);  // both halves of the key pairs
    mbar_init(g_ready, 128);
    mbar_init(s_ready, 128);
    mbar_init(ac_full, 1);
    mbar_init(x_free, 128);
    mbar_init(y_full, 1);
    mbar_init(cb_ready, 128);
    mbar_init(d_full, 1);
    mbar_init(e3_done, 128);
    mbar_init(drain, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&z_full[b], 128);
      mbar_init(&z_empty[b], 256);  // read by both query halves
    }
    mbar_init(k_full, 1);
    mbar_init(v_full, 1);
    mbar_init(kc_ready, 128);
    *abort_word = 0;
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  auto wait = [&](uint64_t *bar, uint32_t parity) { return mbar_wait(bar, parity, abort_word, status); };

  if (warp == 0) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t iKK = idesc_bf16_f32(128, 128, 0, 0);
      constexpr uint32_t iKM = idesc_bf16_f32(128, 128, 0, 1);
      constexpr uint32_t iMM = idesc_bf16_f32(128, 128, 1, 1);
      const uint32_t sKhi = smem_u32(sm + L::Khi), sKlo = smem_u32(sm + L::Klo), sV = smem_u32(sm + L::V),
                     sGhi = smem_u32(sm + L::Ghi), sGlo = smem_u32(sm + L::Glo), sShi = smem_u32(sm + L::Shi),
                     sSlo = smem_u32(sm + L::Slo);
      const uint32_t tS = tmem + kP1S, tQh = tmem + kP1Q, tQl = tmem + kP1Q + 64;
      int k_issued = 1;  // key loads issued (chunk 0's by the QK warps)
      for (int c = 0; c < nloc; ++c) {
        const uint32_t ph = c & 1;
        const uint32_t tX = tmem + p1_ra(c), tCB = tmem + p1_rc(c);
        if (c + 1 < nloc) {  // the next chunk's rows into L2
          const long t1 = (long)(c0 + c + 1) * kC;
          const uint32_t rows = (uint32_t)min((long)kC, N - t1);
          prefetch_l2(qh + t1 * kD, rows * kD * 2);
          prefetch_l2(kh + t1 * kD, rows * kD * 2);
          prefetch_l2(vh + t1 * kD, rows * kD * 2);
          prefetch_l2(gh + t1 * kD, rows * kD * 4);
        }
        // each product waits only for its own operands
        if (!wait(q_ready, ph) || !wait(k_ready, ph)) break;
        tc_fence_after();
        // A = Q K^T (pairs: Qh Kh + Qh Kl + Ql Kh)
#pragma unroll 4
        for (int ks = 0; ks < 8; ++ks) {
          mma_bf16_ts(tX, tQh + 8 * ks, kdesc(sKhi, ks), iKK, ks > 0);
          mma_bf16_ts(tX, tQh + 8 * ks, kdesc(sKlo, ks), iKK, 1);
          mma_bf16_ts(tX, tQl + 8 * ks, kdesc(sKhi, ks), iKK, 1);
        }
        // C goes into the region the previous chunk's dq phase reads
        if (!wait(g_ready, ph) || !wait(v_full, ph) || (c > 0 && !wait(e3_done, (c - 1) & 1))) break;
        tc_fence_after();
        // C = dO V^T
#pragma unroll 4
        for (int ks = 0; ks < 8; ++ks) {
          mma_bf16(tCB, kdesc(sGhi, ks), kdesc(sV, ks), iKK, ks > 0);
          mma_bf16(tCB, kdesc(sGlo, ks), kdesc(sV, ks), iKK, 1);
        }
        mma_commit(ac_full);
        // S += K^T V once the pair copy of S_prev has been taken
        if (!wait(s_ready, ph)) break;
        tc_fence_after();
#pragma unroll 4
        for (int ks = 0; ks < 8; ++ks) {
          mma_bf16(tS, mndesc(sKhi, ks), mndesc(sV, ks), iMM, 1);
          mma_bf16(tS, mndesc(sKlo, ks), mndesc(sV, ks), iMM, 1);
        }
        // Y = dO S_prev^T (S copy rows = features i, K-major over value components), into X once
        // the epilogue has read A from it
        if (!wait(x_free, ph)) break;
        tc_fence_after();
#pragma unroll 4
        for (int ks = 0; ks < 8; ++ks) {
          mma_bf16(tX, kdesc(sGhi, ks), kdesc(sShi, ks), iKK, ks > 0);
          mma_bf16(tX, kdesc(sGhi, ks), kdesc(sSlo, ks), iKK, 1);
          mma_bf16(tX, kdesc(sGlo, ks), kdesc(sShi, ks), iKK, 1);
        }
        mma_commit(y_full);
        if (!wait(cb_ready, ph)) break;
        tc_fence_after();
        // X += B' K: B' from tensor memory (keys [16 ks, 16 ks + 16): 8 columns hi, 8 lo)
#pragma unroll 4
        for (int ks = 0; ks < 8; ++ks) {
          mma_bf16_ts(tX, tCB + 16 * ks, mndesc(sKhi, ks), iKM, 1);
          mma_bf16_ts(tX, tCB + 16 * ks + 8, mndesc(sKhi, ks), iKM, 1);
          mma_bf16_ts(tX, tCB + 16 * ks, mndesc(sKlo, ks), iKM, 1);
        }
        mma_commit(d_full);
        // the next chunk's raw keys as soon as this chunk's products are done with the K tiles
        if (c + 1 < nloc) {
          if (!wait(d_full, ph)) break;
          mbar_arrive_expect_tx(k_full, kTile);
          tma_load_3d(sm + L::Khi, &p.tk, k_full, 0, (c0 + c + 1) * kC, bh);
          tma_load_3d(sm + L::Khi + kBlk, &p.tk, k_full, 64, (c0 + c + 1) * kC, bh);
          k_issued = c + 2;
        }
      }
      mma_commit(drain);
      wait_drain(drain, 0, status);
      // every key load issued must land before shared memory is released (chunk 0's by the QK warps)
      if (nloc > 0) wait_drain(k_full, (uint32_t)(k_issued - 1) & 1, status);
    }
  } else if (warp < kP1WarpG) {
    // ---------------- QK warps: keys, queries, copies of the state ----------------
    const int r = (warp & 3) * 32 + lane;       // tensor-memory lane: chunk row, or state row for the copies
    const int tid = threadIdx.x - 32;           // 0..127
    const uint32_t tl = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    uint8_t *Shi = sm + L::Shi, *Slo = sm + L::Slo;
    uint4 *kt = reinterpret_cast<uint4 *>(sm + L::Khi), *lt = reinterpret_cast<uint4 *>(sm + L::Klo);
    if (tid == 0) {  // chunk 0's raw keys into the Khi tile (the MMA thread loads the later ones)
      prefetch_tmap(&p.tk);
      mbar_arrive_expect_tx(k_full, kTile);
      tma_load_3d(sm + L::Khi, &p.tk, k_full, 0, c0 * kC, bh);
      tma_load_3d(sm + L::Khi + kBlk, &p.tk, k_full, 64, c0 * kC, bh);
    }
    {
      // initial state: S0 plus the sums of the earlier segments (the state pass's pieces), into
      // tensor memory and its pair copy; z0 plus theirs into z buffer 0
      const long npre = (long)seg * p.parts;  // pieces of this head before this segment
      const float *pieces = p.part_S + (long)bh * (p.nseg - 1) * p.parts * kD * kD;
      for (int cb = 0; cb < 8; ++cb) {
        float f[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) f[e] = 0.f;
        if (p.S0) {
          const float4 *src = reinterpret_cast<const float4 *>(p.S0 + ((long)bh * kD + r) * kD + cb * 16);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float4 x = src[e];
            f[4 * e] += x.x, f[4 * e + 1] += x.y, f[4 * e + 2] += x.z, f[4 * e + 3] += x.w;
          }
        }
        for (long pc = 0; pc < npre; ++pc) {
          const float4 *src = reinterpret_cast<const float4 *>(pieces + (pc * kD + r) * kD + cb * 16);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float4 x = src[e];
            f[4 * e] += x.x, f[4 * e + 1] += x.y, f[4 * e + 2] += x.z, f[4 * e + 3] += x.w;
          }
        }
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) w[e] = __float_as_uint(f[e]);
        tmem_st16(tl + kP1S + cb * 16, w);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          uint32_t h[4], l[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) split2(__uint_as_float(w[8 * q + 2 * e]), __uint_as_float(w[8 * q + 2 * e + 1]), h[e], l[e]);
          *tile_chunk(Shi, r, cb * 16 + 8 * q) = make_uint4(h[0], h[1], h[2], h[3]);
          *tile_chunk(Slo, r, cb * 16 + 8 * q) = make_uint4(l[0], l[1], l[2], l[3]);
        }
      }
      float zr = p.z0 ? p.z0[(long)bh * kD + r] : 0.f;
      const float *zpieces = p.part_z + (long)bh * (p.nseg - 1) * p.parts * kD;
      for (long pc = 0; pc < npre; ++pc) zr += zpieces[pc * kD + r];
      zbuf[r] = zr;
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(s_ready);
      mbar_arrive(&z_full[0]);
    }
    bool ok = true;
    // queries 0-63 of chunk c (row r already loaded into x) as phi pairs into tensor memory, once
    // the previous chunk's B' phase has read the phi(Q) columns and chunk c's z is complete
    auto query_pairs = [&](int c, const uint4 (&x)[8], int T) -> bool {
      ok = wait(&z_full[c & 1], (c >> 1) & 1) && (c == 0 || wait(cb_ready, (c - 1) & 1));
      if (bar_or(kBarQK, 128, !ok)) return false;
      tc_fence_after();
      den_x[r] = query_pairs_half(x, r < T, zbuf + (c & 1) * kD, tl, 0);
      mbar_arrive(&z_empty[c & 1]);
      tc_fence_before();
      mbar_arrive(q_ready);
      return true;
    };
    for (int c = 0; c < nloc; ++c) {
      const long t0 = (long)(c0 + c) * kC;
      const int T = (int)min((long)kC, N - t0);
      // chunk 0's queries 0-63, loaded while the keys are transformed (later chunks' are formed
      // in the chunk before)
      uint4 x[8];
      if (c == 0 && r < T) load_row_half(qh + (t0 + r) * kD, x);
      // keys: the raw tile has landed; phi pairs in place (hi) and into Klo (lo), this half of
      // the chunks (the G warps take the other)
      ok = wait(k_full, c & 1);
      if (bar_or(kBarQK, 128, !ok)) break;
      key_pairs(kt, lt, tid, T);
      fence_async_smem();
      mbar_arrive(k_ready);
      if (c == 0 && !query_pairs(0, x, T)) break;
      if (c + 1 == nloc) break;
      // the next chunk's queries, loaded while the state copy is made
      const long t1 = t0 + kC;
      const int T1 = (int)min((long)kC, N - t1);
      if (r < T1) load_row_half(qh + (t1 + r) * kD, x);
      // pair copy of the state the next chunk reads, once this chunk's Y has read the current
      // copy and its S update has completed
      ok = wait(y_full, c & 1);
      if (bar_or(kBarQK, 128, !ok)) break;
      tc_fence_after();
      for (int cb = 0; cb < 8; ++cb) {
        uint32_t w[16];
        tmem_ld16(tl + kP1S + cb * 16, w);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          uint32_t h[4], l[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) split2(__uint_as_float(w[8 * q + 2 * e]), __uint_as_float(w[8 * q + 2 * e + 1]), h[e], l[e]);
          *tile_chunk(Shi, r, cb * 16 + 8 * q) = make_uint4(h[0], h[1], h[2], h[3]);
          *tile_chunk(Slo, r, cb * 16 + 8 * q) = make_uint4(l[0], l[1], l[2], l[3]);
        }
      }
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(s_ready);
      // the next chunk's query pairs as soon as this chunk's B' phase is done
      if (!query_pairs(c + 1, x, T1)) break;
    }
  } else if (warp < kP1WarpE) {
    // ---------------- G warps: dO pairs (coalesced rows), V by TMA ----------------
    const int gt = threadIdx.x - kP1WarpG * 32;  // 0..127
    const int wg = gt >> 5;                       // rows 32 wg .. 32 wg + 31
    uint8_t *Ghi = sm + L::Ghi, *Glo = sm + L::Glo;
    int v_issued = 0;
    if (gt == 0) prefetch_tmap(&p.tv);
    // dO pairs of chunk c and its V (by TMA), once the previous chunk's products are done with
    // those tiles (the caller waits)
    auto dO_pairs = [&](int c) {
      const long t0 = (long)(c0 + c) * kC;
      const int T = (int)min((long)kC, N - t0);
      if (gt == 0) {
        mbar_arrive_expect_tx(v_full, kTile);
        tma_load_3d(sm + L::V, &p.tv, v_full, 0, (int)t0, bh);
        tma_load_3d(sm + L::V + kBlk, &p.tv, v_full, 64, (int)t0, bh);
        v_issued = c + 1;
      }
      // lane l converts features 4l .. 4l + 3 of each row (one 512-byte row per warp load)
      const int col = 4 * lane;
      const uint32_t off = (col >> 6) * kBlk;
#pragma unroll 1
      for (int rr = 0; rr < 32; rr += 16) {  // two rounds of 16 rows in flight
        float4 gg[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int row = 32 * wg + rr + e;
          gg[e] = row < T ? __ldg(reinterpret_cast<const float4 *>(gh + (t0 + row) * kD + col))
                          : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int row = 32 * wg + rr + e;
          uint32_t h0, l0, h1, l1;
          split2(gg[e].x, gg[e].y, h0, l0);
          split2(gg[e].z, gg[e].w, h1, l1);
          const uint32_t o = off + sw128_offset(row, col & 63);
          *reinterpret_cast<uint2 *>(Ghi + o) = make_uint2(h0, h1);
          *reinterpret_cast<uint2 *>(Glo + o) = make_uint2(l0, l1);
        }
      }
      fence_async_smem();
      mbar_arrive(g_ready);
    };
    // queries 64-127 of chunk c (row r already loaded into x) as phi pairs into this warp's
    // tensor-memory lanes, as the QK warps do 0-63
    const int r = (warp & 3) * 32 + lane;
    const uint32_t tl = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    auto query_pairs = [&](int c, const uint4 (&x)[8], int T) -> bool {
      const bool okq = wait(&z_full[c & 1], (c >> 1) & 1) && (c == 0 || wait(cb_ready, (c - 1) & 1));
      if (bar_or(kBarG, 128, !okq)) return false;
      tc_fence_after();
      den_x[kD + r] = query_pairs_half(x, r < T, zbuf + (c & 1) * kD, tl, 1);
      mbar_arrive(&z_empty[c & 1]);
      tc_fence_before();
      mbar_arrive(q_ready);
      return true;
    };
    if (nloc > 0) dO_pairs(0);
    for (int c = 0; c < nloc; ++c) {
      const long t0 = (long)(c0 + c) * kC;
      const int T = (int)min((long)kC, N - t0);
      uint4 x[8];
      if (c == 0 && r < T) load_row_half(qh + (t0 + r) * kD, x, 1);
      // the other half of this chunk's key pairs, then its key column sums (for the E warps' z)
      bool okk = wait(k_full, c & 1);
      if (bar_or(kBarG, 128, !okk)) break;
      key_pairs(reinterpret_cast<uint4 *>(sm + L::Khi), reinterpret_cast<uint4 *>(sm + L::Klo), 128 + gt, T);
      fence_async_smem();
      mbar_arrive(k_ready);
      if (c == 0 && !query_pairs(0, x, T)) break;
      // this chunk's key column sums, for the E warps' z (both halves of the pairs are written)
      okk = wait(k_ready, c & 1);
      if (bar_or(kBarG, 128, !okk)) break;
      const float2 cs = pair_column_sums(sm + L::Khi, sm + L::Klo, gt, T);
      if (lane < 16) {
        const int pc = 2 * ((gt & 15) + 16 * (gt >> 5));
        kcol[pc] = cs.x;
        kcol[pc + 1] = cs.y;
      }
      mbar_arrive(kc_ready);
      if (c + 1 == nloc) break;
      // the next chunk: its queries (loaded first), its dO pairs and V once this chunk's Y has
      // read the tiles, then its query pairs once this chunk's B' phase is done
      const long t1 = t0 + kC;
      const int T1 = (int)min((long)kC, N - t1);
      if (r < T1) load_row_half(qh + (t1 + r) * kD, x, 1);
      okk = wait(y_full, c & 1);
      if (bar_or(kBarG, 128, !okk)) break;
      dO_pairs(c + 1);
      if (!query_pairs(c + 1, x, T1)) break;
    }
    if (gt == 0 && v_issued > 0) wait_drain(v_full, (v_issued - 1) & 1, status);
  } else {
    // ---------------- E warps: scores, den, gden, B', the next chunk's z, dq ----------------
    const int t = (warp & 3) * 32 + lane;  // tensor-memory lane = chunk row; also feature t of z
    const uint32_t tl = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    for (int c = 0; c < nloc; ++c) {
      const long t0 = (long)(c0 + c) * kC;
      const int T = (int)min((long)kC, N - t0);
      const int jmax = min(t, T - 1);  // keys kept: j <= t and j < T
      const uint32_t rA = tl + p1_ra(c), rC = tl + p1_rc(c);
      uint32_t ra[32], rc[32];
      // E1: row sums of A and of A * C
      bool ok = wait(q_ready, c & 1) && wait(k_ready, c & 1) && wait(ac_full, c & 1);
      if (bar_or(kBarE, 128, !ok)) break;
      tc_fence_after();
      float rs = 0.f, ac = 0.f;
#pragma unroll 1
      for (int cb = 0; cb < 4; ++cb) {
        tmem_ld32x2(rA + cb * 32, rC + cb * 32, ra, rc);
#pragma unroll
        for (int m = 0; m < 32; ++m) {
          const float a = cb * 32 + m <= jmax ? __uint_as_float(ra[m]) : 0.f;
          rs += a;
          ac = fmaf(a, __uint_as_float(rc[m]), ac);
        }
      }
      const float den = ((den_x[t] + den_x[kD + t]) + rs) + p.eps;
      tc_fence_before();
      mbar_arrive(x_free);
      // E2: gden from phi(q) . Y, the next chunk's z, then B' = C + den gden in place as bf16 pairs
      ok = wait(y_full, c & 1);
      if (bar_or(kBarE, 128, !ok)) break;
      tc_fence_after();
      float qy = 0.f;
#pragma unroll 1
      for (int b = 0; b < 4; ++b) {
        uint32_t qhw[16], qlw[16];
        tmem_ld32_16x2(rA + b * 32, tl + kP1Q + 16 * b, tl + kP1Q + 64 + 16 * b, ra, qhw, qlw);
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          qy = fmaf(lo16(qhw[m]) + lo16(qlw[m]), __uint_as_float(ra[2 * m]), qy);
          qy = fmaf(hi16(qhw[m]) + hi16(qlw[m]), __uint_as_float(ra[2 * m + 1]), qy);
        }
      }
      const float gden = -((qy + ac) / den) / den;
      const float dg = den * gden;
      // this chunk's key column sums (waited for here, before cb_ready, so that the G warps
      // cannot complete the next chunk's before this wait)
      ok = wait(kc_ready, c & 1);
      if (bar_or(kBarE, 128, !ok)) break;
      const float *z = zbuf + (c & 1) * kD;
      // z for the next chunk: z_prev plus this chunk's key column sums (thread t owns feature t),
      // before the next chunk's query pairs need it; the previous reads of that buffer (the
      // query pairs and this group's dq of the chunk before) are done
      if (c + 1 < nloc) {
        const int nb = (c + 1) & 1;
        ok = c + 1 < 2 || wait(&z_empty[nb], (((c + 1) >> 1) - 1) & 1);
        if (bar_or(kBarE, 128, !ok)) break;
        zbuf[nb * kD + t] = z[t] + kcol[t];
        mbar_arrive(&z_full[nb]);
      }
#pragma unroll 1
      for (int cb = 0; cb < 4; cb += 2) {
        tmem_ld32x2(rC + cb * 32, rC + cb * 32 + 32, ra, rc);
        split_scores32(ra, cb, [&](int j) { return j <= jmax; }, [&](int, float x) { return x + dg; });
        split_scores32(rc, cb + 1, [&](int j) { return j <= jmax; }, [&](int, float x) { return x + dg; });
        tmem_st32(rC + cb * 32, ra);
        tmem_st32(rC + cb * 32 + 32, rc);
      }
      tc_fence_before();
      mbar_arrive(cb_ready);
      // E3: dq = ((Y + B' K) / den + gden z_prev) phi'(q), phi'(q) = min(phi(q), 1) from the
      // query row itself (the next chunk's pairs may already fill the phi(Q) columns)
      const uint8_t *qrow = reinterpret_cast<const uint8_t *>(qh + (t0 + t) * kD);
      uint32_t na[8], nb8[8];  // the next 32 features' query words
      auto load_q = [&](int b) {
        if (t < T) {
          ld_row32(qrow + 64 * b, na);
          ld_row32(qrow + 64 * b + 32, nb8);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) na[e] = nb8[e] = 0u;
        }
      };
      load_q(0);
      ok = wait(d_full, c & 1);
      if (bar_or(kBarE, 128, !ok)) break;
      tc_fence_after();
      const float inv = 1.f / den;
      float *dst = p.dq + ((long)bh * N + t0 + t) * kD;
#pragma unroll 1
      for (int b = 0; b < 4; ++b) {
        uint32_t qw[16];
#pragma unroll
        for (int e = 0; e < 8; ++e) qw[e] = na[e], qw[8 + e] = nb8[e];
        if (b < 3) load_q(b + 1);
        tmem_ld32(rA + b * 32, ra);
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          const float2 f = phi2(lo16(qw[m]), hi16(qw[m]));
          const float f0 = fminf(f.x, 1.f), f1 = fminf(f.y, 1.f);
          ra[2 * m] = __float_as_uint(fmaf(__uint_as_float(ra[2 * m]), inv, z[32 * b + 2 * m] * gden) * f0);
          ra[2 * m + 1] =
              __float_as_uint(fmaf(__uint_as_float(ra[2 * m + 1]), inv, z[32 * b + 2 * m + 1] * gden) * f1);
        }
        if (t < T) {
#pragma unroll
          for (int e = 0; e < 4; ++e) st_row32(dst + 32 * b + 8 * e, ra + 8 * e);
        }
      }
      if (t < T) {
        p.den[(long)bh * N + t0 + t] = den;
        p.gden[(long)bh * N + t0 + t] = gden;
      }
      tc_fence_before();
      mbar_arrive(e3_done);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// Pass 2: chunks in reverse, U (and u) carried; role 0 dv, role 1 dk.
// ---------------------------------------------------------------------------
// Shared memory: phi(Q), gnum and the copy of U as bf16 pairs (six tiles,
// 192 KB), a staging tile for the next chunk's raw queries (32 KB), the
// chunk's gden, the carried u (role 1), barriers.
struct P2Layout {
  static constexpr uint32_t Qhi = 0, Qlo = kTile, Nhi = 2 * kTile, Nlo = 3 * kTile, Uhi = 4 * kTile, Ulo = 5 * kTile,
                            Kst = 6 * kTile;
  static constexpr uint32_t Gd = 7 * kTile;  // [128] gden of the chunk
  static constexpr uint32_t Ub = Gd + 512;   // [128] u carried into the chunk (role 1)
  static constexpr uint32_t Bars = Ub + 512;
  static constexpr int kNumBars = 14;
  static constexpr uint32_t Misc = Bars + kNumBars * 8;
  static constexpr uint32_t Bytes = Misc + 16;
};
static_assert(P2Layout::Bytes <= 232448, "pass 2 shared memory");

// TMEM columns of pass 2: U accumulator; X = the key-side scores (role 0:
// K Q^T, role 1: V gnum^T), then as bf16 pairs; O = dv or dk; the key operand
// (role 0: phi(K) as pairs, 128 columns; role 1: V, 64 columns, then the raw
// keys for phi'(k), 64 columns).
constexpr uint32_t kP2U = 0, kP2X = 128, kP2O = 256, kP2K = 384;

// Warp roles of pass 2 (13 warps): 0 MMA issuer; 1-4 key operand (rows into
// tensor memory), copies of U; 5-8 gnum pairs (coalesced rows), gden and the
// phi(Q) pairs from the staged raw queries; 9-12 scores and outputs.
constexpr int kP2Threads = 416;
constexpr int kP2WarpN = 5, kP2WarpE = 9;

// phi pairs of the staged raw query tile into the Q tiles (same swizzled
// layout): thread u of 256 takes chunks u + 256 i; rows past T are zeros.
__device__ __forceinline__ void query_pairs_staged(uint8_t *sm, int u, int T) {
  const uint4 *raw = reinterpret_cast<const uint4 *>(sm + P2Layout::Kst);
  uint4 *hi = reinterpret_cast<uint4 *>(sm + P2Layout::Qhi), *lo = reinterpret_cast<uint4 *>(sm + P2Layout::Qlo);
#pragma unroll 4
  for (int i = 0; i < 8; ++i) {
    const int ch = u + 256 * i;
    uint4 h = make_uint4(0u, 0u, 0u, 0u), l = h;
    if (((ch & 1023) >> 3) < T) phi_pair8(raw[ch], h, l);
    hi[ch] = h;
    lo[ch] = l;
  }
}

template <int kRole>
__device__ __forceinline__ void pass2_role(const BwdTcParams &p) {
  using L = P2Layout;
  constexpr bool kDk = kRole == 1;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) atomicOr(&g_bwd_status, kAbortMisaligned);
    return;
  }
  uint8_t *sm = smem_raw;
  float *gd = reinterpret_cast<float *>(sm + L::Gd);
  float *ub = reinterpret_cast<float *>(sm + L::Ub);
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::Bars);
  uint64_t *q_ready = bars + 0, *k_ready = bars + 1, *n_ready = bars + 2, *u_ready = bars + 3, *x_full = bars + 4,
           *x_split = bars + 5, *o_full = bars + 6, *o_done = bars + 7, *drain = bars + 8, *q_full = bars + 9,
           *q_used = bars + 10,
           *u_done = bars + 11,  // the chunk's U update complete: its operand tiles and U are free
           *ucol_done = bars + 12,  // role 1: the epilogue's read of the Q tiles and gd for u is done
           *kp_ready = bars + 13;   // role 1: the chunk's raw keys are in tensor memory
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + L::Misc);
  volatile uint32_t *abort_word = reinterpret_cast<volatile uint32_t *>(sm + L::Misc + 4);
  unsigned int *status = &g_bwd_status;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.x;
  const long N = p.N;
  const int nch = (int)((N + kC - 1) / kC);
  const __nv_bfloat16 *qh = p.q + (long)bh * N * kD, *kh = p.k + (long)bh * N * kD, *vh = p.v + (long)bh * N * kD;
  const float *gh = p.dout + (long)bh * N * kD;

  if (threadIdx.x == 0) {
    mbar_init(q_ready, 256);  // both halves of the query pairs
    mbar_init(k_ready, 128);
    mbar_init(n_ready, 128);
    mbar_init(u_ready, 128);
    mbar_init(x_full, 1);
    mbar_init(x_split, 128);
    mbar_init(o_full, 1);
    mbar_init(u_done, 1);
    mbar_init(ucol_done, 128);
    mbar_init(kp_ready, 128);
    mbar_init(o_done, 128);
    mbar_init(drain, 1);
    mbar_init(q_full, 1);
    mbar_init(q_used, 256);
    *abort_word = 0;
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  auto wait = [&](uint64_t *bar, uint32_t parity) { return mbar_wait(bar, parity, abort_word, status); };

  if (warp == 0) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t iKK = idesc_bf16_f32(128, 128, 0, 0);
      constexpr uint32_t iKM = idesc_bf16_f32(128, 128, 0, 1);
      constexpr uint32_t iMM = idesc_bf16_f32(128, 128, 1, 1);
      const uint32_t sQhi = smem_u32(sm + L::Qhi), sQlo = smem_u32(sm + L::Qlo), sNhi = smem_u32(sm + L::Nhi),
                     sNlo = smem_u32(sm + L::Nlo), sUhi = smem_u32(sm + L::Uhi), sUlo = smem_u32(sm + L::Ulo);
      const uint32_t tU = tmem + kP2U, tX = tmem + kP2X, tO = tmem + kP2O, tKh = tmem + kP2K,
                     tKl = tmem + kP2K + 64;
      for (int it = 0; it < nch; ++it) {
        const int c = nch - 1 - it;
        const uint32_t ph = it & 1;
        if (c > 0) {  // the next chunk's rows into L2
          const long t1 = (long)(c - 1) * kC;
          prefetch_l2(qh + t1 * kD, kC * kD * 2);
          prefetch_l2(kDk ? vh + t1 * kD : kh + t1 * kD, kC * kD * 2);
          if (kDk) prefetch_l2(kh + t1 * kD, kC * kD * 2);
          prefetch_l2(gh + t1 * kD, kC * kD * 4);
        }
        // X needs only the key operand and one other: the query pairs (role 0, X = K Q^T) or the
        // gnum pairs (role 1, X = V gnum^T); the remaining one is waited for before O += X B
        if (!wait(k_ready, ph) || !wait(kDk ? n_ready : q_ready, ph)) break;
        tc_fence_after();
        if (!kDk) {
          // X = K Q^T (rows keys j, columns queries t)
#pragma unroll 4
          for (int ks = 0; ks < 8; ++ks) {
            mma_bf16_ts(tX, tKh + 8 * ks, kdesc(sQhi, ks), iKK, ks > 0);
            mma_bf16_ts(tX, tKh + 8 * ks, kdesc(sQlo, ks), iKK, 1);
            mma_bf16_ts(tX, tKl + 8 * ks, kdesc(sQhi, ks), iKK, 1);
          }
        } else {
          // X = V gnum^T
#pragma unroll 4
          for (int ks = 0; ks < 8; ++ks) {
            mma_bf16_ts(tX, tKh + 8 * ks, kdesc(sNhi, ks), iKK, ks > 0);
            mma_bf16_ts(tX, tKh + 8 * ks, kdesc(sNlo, ks), iKK, 1);
          }
        }
        mma_commit(x_full);  // the epilogue splits X while O = K U (or V U^T) runs
        if (!wait(u_ready, ph) || (it > 0 && !wait(o_done, (it - 1) & 1))) break;
        tc_fence_after();
        if (!kDk) {
          // O = K U (U rows = features i: the K index)
#pragma unroll 4
          for (int ks = 0; ks < 8; ++ks) {
            mma_bf16_ts(tO, tKh + 8 * ks, mndesc(sUhi, ks), iKM, ks > 0);
            mma_bf16_ts(tO, tKh + 8 * ks, mndesc(sUlo, ks), iKM, 1);
            mma_bf16_ts(tO, tKl + 8 * ks, mndesc(sUhi, ks), iKM, 1);
          }
        } else {
          // O = V U^T (U rows = features i: the N index, K-major over value components)
#pragma unroll 4
          for (int ks = 0; ks < 8; ++ks) {
            mma_bf16_ts(tO, tKh + 8 * ks, kdesc(sUhi, ks), iKK, ks > 0);
            mma_bf16_ts(tO, tKh + 8 * ks, kdesc(sUlo, ks), iKK, 1);
          }
        }
        if (!wait(kDk ? q_ready : n_ready, ph)) break;
        tc_fence_after();
        // U += Q^T gnum, before O += X B: its commit frees the key operand, U and (role 0) the
        // query pairs or (role 1) the gnum pairs for the next chunk while O += X B still runs
#pragma unroll 4
        for (int ks = 0; ks < 8; ++ks) {
          mma_bf16(tU, mndesc(sQhi, ks), mndesc(sNhi, ks), iMM, 1);
          mma_bf16(tU, mndesc(sQhi, ks), mndesc(sNlo, ks), iMM, 1);
          mma_bf16(tU, mndesc(sQlo, ks), mndesc(sNhi, ks), iMM, 1);
        }
        mma_commit(u_done);
        if (!wait(x_split, ph)) break;
        tc_fence_after();
        // O += X B with X from tensor memory as pairs (queries [16 ks, 16 ks + 16): 8 columns hi,
        // 8 lo) and B = gnum (role 0) or phi(Q) (role 1), rows = queries; its commit also frees B
        const uint32_t sBhi = kDk ? sQhi : sNhi, sBlo = kDk ? sQlo : sNlo;
#pragma unroll 4
        for (int ks = 0; ks < 8; ++ks) {
          mma_bf16_ts(tO, tX + 16 * ks, mndesc(sBhi, ks), iKM, 1);
          mma_bf16_ts(tO, tX + 16 * ks + 8, mndesc(sBhi, ks), iKM, 1);
          mma_bf16_ts(tO, tX + 16 * ks, mndesc(sBlo, ks), iKM, 1);
        }
        mma_commit(o_full);
      }
      mma_commit(drain);
      wait_drain(drain, 0, status);
    }
  } else if (warp < kP2WarpN) {
    // ---------------- QK warps: key operand into tensor memory, copies of U ----------------
    const int r = (warp & 3) * 32 + lane;  // tensor-memory lane: chunk row, or state row of U
    const uint32_t tl = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    uint8_t *Uhi = sm + L::Uhi, *Ulo = sm + L::Ulo;
    const __nv_bfloat16 *key = kDk ? vh : kh;
    {
      // U at the end of the sequence: dS (or zero) into tensor memory and its pair copy
      for (int cb = 0; cb < 8; ++cb) {
        uint32_t w[16];
        if (p.dS) {
          const float4 *src = reinterpret_cast<const float4 *>(p.dS + ((long)bh * kD + r) * kD + cb * 16);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float4 f = src[e];
            w[4 * e] = __float_as_uint(f.x), w[4 * e + 1] = __float_as_uint(f.y);
            w[4 * e + 2] = __float_as_uint(f.z), w[4 * e + 3] = __float_as_uint(f.w);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) w[e] = 0u;
        }
        tmem_st16(tl + kP2U + cb * 16, w);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          uint32_t h[4], l[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) split2(__uint_as_float(w[8 * q + 2 * e]), __uint_as_float(w[8 * q + 2 * e + 1]), h[e], l[e]);
          *tile_chunk(Uhi, r, cb * 16 + 8 * q) = make_uint4(h[0], h[1], h[2], h[3]);
          *tile_chunk(Ulo, r, cb * 16 + 8 * q) = make_uint4(l[0], l[1], l[2], l[3]);
        }
      }
    }
    bool ok = true;
    for (int it = 0; it < nch; ++it) {
      const int c = nch - 1 - it;
      const long t0 = (long)c * kC;
      const int T = (int)min((long)kC, N - t0);
      // this row of the key operand, loaded while the previous chunk's products finish
      uint4 x[16];
      if (r < T) {
        load_row_half(key + (t0 + r) * kD, *reinterpret_cast<uint4 (*)[8]>(&x[0]), 0);
        load_row_half(key + (t0 + r) * kD, *reinterpret_cast<uint4 (*)[8]>(&x[8]), 1);
      }
      ok = it == 0 || wait(u_done, (it - 1) & 1);
      if (bar_or(kBarQK, 128, !ok)) break;
      tc_fence_after();
      // key operand, row r: role 0 phi(k) pairs (hi columns 0-63, lo 64-127), role 1 v as given;
      // rows past the end are zeros
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const uint4 xe = r < T ? x[e] : make_uint4(0u, 0u, 0u, 0u);
        if (!kDk) {
          uint4 h = make_uint4(0u, 0u, 0u, 0u), l = h;
          if (r < T) phi_pair8(xe, h, l);
          tmem_st4_nowait(tl + kP2K + 4 * e, h.x, h.y, h.z, h.w);
          tmem_st4_nowait(tl + kP2K + 64 + 4 * e, l.x, l.y, l.z, l.w);
        } else {
          tmem_st4_nowait(tl + kP2K + 4 * e, xe.x, xe.y, xe.z, xe.w);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(k_ready);
      // the pair copy of U (every chunk after this one folded in); the tiles were last read by
      // the previous chunk's products, which have completed
      auto copy_u = [&]() {
        if (it == 0) return;
        for (int cb = 0; cb < 8; ++cb) {
          uint32_t w[16];
          tmem_ld16(tl + kP2U + cb * 16, w);
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            uint32_t h[4], l[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) split2(__uint_as_float(w[8 * q + 2 * e]), __uint_as_float(w[8 * q + 2 * e + 1]), h[e], l[e]);
            *tile_chunk(Uhi, r, cb * 16 + 8 * q) = make_uint4(h[0], h[1], h[2], h[3]);
            *tile_chunk(Ulo, r, cb * 16 + 8 * q) = make_uint4(l[0], l[1], l[2], l[3]);
          }
        }
      };
      // half of the phi(Q) pairs from the staged raw queries (the N warps take the other half)
      auto query_half = [&]() -> bool {
        // role 1: the epilogue reads the previous chunk's query pairs for u after its split, and
        // they are the B operand of that chunk's O += X Q
        ok = wait(q_full, it & 1) &&
             (!kDk || it == 0 || (wait(ucol_done, (it - 1) & 1) && wait(o_full, (it - 1) & 1)));
        if (bar_or(kBarQK, 128, !ok)) return false;
        query_pairs_staged(sm, threadIdx.x - 32, T);
        fence_async_smem();
        mbar_arrive(q_ready);
        mbar_arrive(q_used);  // this half is done with the staging tile
        return true;
      };
      // role 0's first product X = K Q^T takes the query pairs; role 1's, X = V gnum^T, does not
      if (!kDk && !query_half()) break;
      copy_u();
      fence_async_smem();
      mbar_arrive(u_ready);
      if (kDk) {
        if (!query_half()) break;
        // role 1: the chunk's raw key rows for phi'(k), into the key-operand columns V leaves
        // free, once the epilogue has read the previous chunk's
        uint4 kx[16];
        if (r < T) {
          load_row_half(kh + (t0 + r) * kD, *reinterpret_cast<uint4 (*)[8]>(&kx[0]), 0);
          load_row_half(kh + (t0 + r) * kD, *reinterpret_cast<uint4 (*)[8]>(&kx[8]), 1);
        }
        ok = it == 0 || wait(o_done, (it - 1) & 1);
        if (bar_or(kBarQK, 128, !ok)) break;
        tc_fence_after();
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const uint4 xe = r < T ? kx[e] : make_uint4(0u, 0u, 0u, 0u);
          tmem_st4_nowait(tl + kP2K + 64 + 4 * e, xe.x, xe.y, xe.z, xe.w);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(kp_ready);
      }
    }
    // role 0: the initial state's gradient dS0 = U after the first chunk
    if (!kDk && p.dS0) {
      ok = ok && wait(u_done, (nch - 1) & 1);
      if (!bar_or(kBarQK, 128, !ok) && !*abort_word) {
        tc_fence_after();
        float *dst = p.dS0 + ((long)bh * kD + r) * kD;
        for (int cb = 0; cb < 4; ++cb) {
          uint32_t w[32];
          tmem_ld32(tl + kP2U + cb * 32, w);
          float4 *d4 = reinterpret_cast<float4 *>(dst + cb * 32);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            d4[e] = make_float4(__uint_as_float(w[4 * e]), __uint_as_float(w[4 * e + 1]), __uint_as_float(w[4 * e + 2]),
                                __uint_as_float(w[4 * e + 3]));
        }
      }
    }
  } else if (warp < kP2WarpE) {
    // ---------------- N warps: gnum = dO / den as pairs (coalesced rows), gden, phi(Q) pairs ----------------
    const int gt = threadIdx.x - kP2WarpN * 32;  // 0..127
    const int wg = gt >> 5;                       // rows 32 wg .. 32 wg + 31
    uint8_t *Nhi = sm + L::Nhi, *Nlo = sm + L::Nlo;
    const int col = 4 * lane;
    const uint32_t off = (col >> 6) * kBlk;
    int q_issued = 0;
    auto load_q = [&](int c) {  // raw queries of chunk c into the staging tile
      mbar_arrive_expect_tx(q_full, kTile);
      tma_load_3d(sm + L::Kst, &p.tq, q_full, 0, c * kC, bh);
      tma_load_3d(sm + L::Kst + kBlk, &p.tq, q_full, 64, c * kC, bh);
      ++q_issued;
    };
    if (gt == 0) {
      prefetch_tmap(&p.tq);
      load_q(nch - 1);
    }
    for (int it = 0; it < nch; ++it) {
      const int c = nch - 1 - it;
      const long t0 = (long)c * kC;
      const int T = (int)min((long)kC, N - t0);
      // this thread's row 32 wg + lane: its gden, and 1 / den broadcast over the warp below
      const int myrow = 32 * wg + lane;
      const float inv_mine = myrow < T ? 1.f / p.den[(long)bh * N + t0 + myrow] : 0.f;
      const float gdn = myrow < T ? p.gden[(long)bh * N + t0 + myrow] : 0.f;
      // gnum rows in two rounds of 16; dO is an input, so where gnum is needed first (role 1)
      // the first round's loads go out before the wait for the previous chunk's products (which
      // still read the N tiles)
      float4 gg[16];
      auto load_round = [&](int rr) {
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int row = 32 * wg + rr + e;
          gg[e] = row < T ? __ldg(reinterpret_cast<const float4 *>(gh + (t0 + row) * kD + col))
                          : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      };
      auto store_round = [&](int rr) {
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int row = 32 * wg + rr + e;
          const float inv = __shfl_sync(0xffffffffu, inv_mine, rr + e);
          uint32_t h0, l0, h1, l1;
          split2(gg[e].x * inv, gg[e].y * inv, h0, l0);
          split2(gg[e].z * inv, gg[e].w * inv, h1, l1);
          const uint32_t o = off + sw128_offset(row, col & 63);
          *reinterpret_cast<uint2 *>(Nhi + o) = make_uint2(h0, h1);
          *reinterpret_cast<uint2 *>(Nlo + o) = make_uint2(l0, l1);
        }
      };
      auto gnum_rest = [&]() {  // round 0 already loaded
        store_round(0);
        load_round(16);
        store_round(16);
        gd[myrow] = gdn;
        fence_async_smem();
        mbar_arrive(n_ready);
      };
      // phi(Q) pairs from the staged raw queries (same swizzled layout), then the next chunk's
      // raw queries into the staging tile once both halves are done with it
      auto query_half = [&]() -> bool {
        // role 1: the previous chunk's query pairs are the B operand of its O += X Q
        bool okq = wait(q_full, it & 1) && (!kDk || it == 0 || wait(o_full, (it - 1) & 1));
        if (bar_or(kBarG, 128, !okq)) return false;
        query_pairs_staged(sm, 128 + gt, T);
        fence_async_smem();
        mbar_arrive(q_ready);
        mbar_arrive(q_used);
        okq = true;
        if (gt == 0 && c > 0) okq = wait(q_used, it & 1);
        if (bar_or(kBarG, 128, !okq)) return false;
        if (gt == 0 && c > 0) load_q(c - 1);
        return true;
      };
      if (kDk) {
        // role 1: X = V gnum^T comes first
        load_round(0);
        // the epilogue's read of gd (and of the query pairs) for u must be done before gd changes
        const bool ok = it == 0 || (wait(u_done, (it - 1) & 1) && wait(ucol_done, (it - 1) & 1));
        if (bar_or(kBarG, 128, !ok)) break;
        gnum_rest();
        if (!query_half()) break;
      } else {
        // role 0: X = K Q^T comes first; gnum is first needed by the U update, and the previous
        // chunk's gnum pairs are the B operand of its O += X gnum
        const bool ok = it == 0 || wait(u_done, (it - 1) & 1);
        if (bar_or(kBarG, 128, !ok)) break;
        if (!query_half()) break;
        load_round(0);
        const bool okn = it == 0 || wait(o_full, (it - 1) & 1);
        if (bar_or(kBarG, 128, !okn)) break;
        gnum_rest();
      }
    }
    if (gt == 0 && q_issued > 0) wait_drain(q_full, (q_issued - 1) & 1, status);
  } else {
    // ---------------- E warps: key-side scores as pairs, then dv or dk ----------------
    const int j = (warp & 3) * 32 + lane;  // tensor-memory lane = key row (or feature, for u)
    const uint32_t tl = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    if (kDk) {
      ub[j] = p.dz ? p.dz[(long)bh * kD + j] : 0.f;
      named_bar(kBarE, 128);
    }
    const uint8_t *Qhi = sm + L::Qhi, *Qlo = sm + L::Qlo;
    bool ok = true;
    for (int it = 0; it < nch; ++it) {
      const int c = nch - 1 - it;
      const long t0 = (long)c * kC;
      const int T = (int)min((long)kC, N - t0);
      ok = wait(x_full, it & 1) && wait(n_ready, it & 1) && wait(q_ready, it & 1);
      if (bar_or(kBarE, 128, !ok)) break;
      tc_fence_after();
      // queries t >= j of the chunk's valid rows (none when the key row itself is past the end)
      const int tmin = j, tend = j < T ? T : 0;
#pragma unroll 1
      for (int cb = 0; cb < 4; cb += 2) {
        uint32_t rx[32], ry[32];
        tmem_ld32x2(tl + kP2X + cb * 32, tl + kP2X + cb * 32 + 32, rx, ry);
        split_scores32(rx, cb, [&](int t) { return t >= tmin && t < tend; },
                       [&](int t, float x) { return kDk ? x + gd[t] : x; });
        split_scores32(ry, cb + 1, [&](int t) { return t >= tmin && t < tend; },
                       [&](int t, float x) { return kDk ? x + gd[t] : x; });
        tmem_st32(tl + kP2X + cb * 32, rx);
        tmem_st32(tl + kP2X + cb * 32 + 32, ry);
      }
      tc_fence_before();
      mbar_arrive(x_split);
      float ucol = 0.f;
      if (kDk) {
        // this chunk's share of u for feature j: sum over its queries of phi(q_t)_j gden_t, read
        // while O += X Q and the U update run (the operand warps wait for ucol_done before they
        // overwrite the query pairs or gd)
        const uint8_t *bh_ = Qhi + (j >> 6) * kBlk, *bl_ = Qlo + (j >> 6) * kBlk;
#pragma unroll 4
        for (int t = 0; t < T; ++t) {
          const uint32_t off = sw128_offset(t, j & 63);
          const float f = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(bh_ + off)) +
                          __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(bl_ + off));
          ucol = fmaf(f, gd[t], ucol);
        }
        mbar_arrive(ucol_done);
      }
      ok = wait(o_full, it & 1) && (!kDk || wait(kp_ready, it & 1));
      if (bar_or(kBarE, 128, !ok)) break;
      tc_fence_after();
      float *dst = (kDk ? p.dk : p.dv) + ((long)bh * N + t0 + j) * kD;
#pragma unroll 1
      for (int b = 0; b < 4; ++b) {
        uint32_t ro[32];
        tmem_ld32(tl + kP2O + b * 32, ro);
        if (kDk) {
          // dk = (V U^T + B Q + u) phi'(k), phi'(x) = 1 above zero, e^x below; the keys of
          // features [32 b, 32 b + 32) from tensor memory (zeros past the end)
          uint32_t kw[16];
          tmem_ld16(tl + kP2K + 64 + 16 * b, kw);
#pragma unroll
          for (int e = 0; e < 2; ++e) {
#pragma unroll
            for (int m = 0; m < 8; ++m) {
              const int col = 32 * b + 16 * e + 2 * m;
              const float2 f = phi2(lo16(kw[8 * e + m]), hi16(kw[8 * e + m]));
              const float da = fminf(f.x, 1.f), db = fminf(f.y, 1.f);
              ro[16 * e + 2 * m] = __float_as_uint((__uint_as_float(ro[16 * e + 2 * m]) + ub[col]) * da);
              ro[16 * e + 2 * m + 1] = __float_as_uint((__uint_as_float(ro[16 * e + 2 * m + 1]) + ub[col + 1]) * db);
            }
          }
        }
        if (j < T) {
#pragma unroll
          for (int e = 0; e < 4; ++e) st_row32(dst + 32 * b + 8 * e, ro + 8 * e);
        }
      }
      if (kDk) {
        named_bar(kBarE, 128);  // every read of u for this chunk is done
        ub[j] += ucol;
      }
      tc_fence_before();
      mbar_arrive(o_done);
    }
    if (kDk && p.dz0) {
      named_bar(kBarE, 128);
      if (ok && !*abort_word) p.dz0[(long)bh * kD + j] = ub[j];
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Both roles of a head run side by side: blockIdx.y = 0 dv, 1 dk.
__global__ void __launch_bounds__(kP2Threads, 1) bwd_pass2_tc(const __grid_constant__ BwdTcParams p) {
  if (blockIdx.y == 0)
    pass2_role<0>(p);
  else
    pass2_role<1>(p);
}

}  // namespace

// [BH][N][128] bf16 as a 3-D tensor; boxes of 64 features x 128 tokens x 1 head, 128-byte swizzle.
bool make_bf16_map(CUtensorMap *m, const void *base, long BH, long N) {
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)N * kD * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)kC, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool backward_tc_supported(const BackwardProblem &b) {
  const Problem &p = b.p;
  const DeviceInfo di = device_info(-1);
  // rows are read and written 32 bytes at a time
  const void *rows[5] = {p.q, p.k, b.dq, b.dk, b.dv};
  for (const void *r : rows)
    if (reinterpret_cast<uintptr_t>(r) & 31u) return false;
  return p.dt == LA_BF16 && p.dk == kD && p.dv == kD && p.N >= 1 && p.N <= 0x7fffffffL && p.BH <= 65535 &&
         di.cc_major == 10 && di.cc_minor == 3 && tensor_map_encoder() != nullptr;
}

cudaError_t launch_causal_backward_tc(const BackwardProblem &b) {
  const Problem &p = b.p;
  cudaError_t e = ensure_smem_optin((const void *)bwd_pass1_tc, (int)P1Layout::Bytes);
  if (e == cudaSuccess) e = ensure_smem_optin((const void *)bwd_pass2_tc, (int)P2Layout::Bytes);
  if (e == cudaSuccess) e = ensure_smem_optin((const void *)bwd_state_tc, (int)StLayout::Bytes);
  if (e != cudaSuccess) return e;
  // pass 1's segments: enough CTAs to cover the SMs once, at least 4 chunks each; the state pass
  // sums each earlier segment in `parts` pieces, enough CTAs to cover the SMs about once
  const long sms = std::max(1, device_info(-1).sm_count);
  const long nch = (p.N + kC - 1) / kC;
  long G = std::max(1L, std::min(sms / p.BH, nch / 4));
  const long seg_chunks = (nch + G - 1) / G;
  G = (nch + seg_chunks - 1) / seg_chunks;
  const long parts = G > 1 ? std::max(1L, std::min(seg_chunks, sms / (p.BH * (G - 1)))) : 1;
  const size_t npieces = (size_t)p.BH * (G - 1) * parts;
  // scratch: den and gden of every token (pass 1 -> pass 2), then the state pass's pieces
  // (each block starts on a 256-byte boundary)
  const size_t dg_f = (2 * (size_t)p.BH * p.N + 63) / 64 * 64;
  const size_t piece_f = npieces * (kD * kD + kD);
  float *scratch = nullptr;
  e = cudaMallocAsync(reinterpret_cast<void **>(&scratch), sizeof(float) * (dg_f + piece_f), p.stream);
  if (e != cudaSuccess) return e;
  BwdTcParams a;
  memset(&a, 0, sizeof a);
  if (!make_bf16_map(&a.tq, p.q, p.BH, p.N) || !make_bf16_map(&a.tk, p.k, p.BH, p.N) ||
      !make_bf16_map(&a.tv, p.v, p.BH, p.N)) {
    cudaFreeAsync(scratch, p.stream);
    return cudaErrorInvalidValue;
  }
  a.q = static_cast<const __nv_bfloat16 *>(p.q);
  a.k = static_cast<const __nv_bfloat16 *>(p.k);
  a.v = static_cast<const __nv_bfloat16 *>(p.v);
  a.dout = b.dout, a.S0 = b.S0, a.z0 = b.z0, a.dS = b.dS, a.dz = b.dz;
  a.dq = b.dq, a.dk = b.dk, a.dv = b.dv, a.dS0 = b.dS0, a.dz0 = b.dz0;
  a.den = scratch;
  a.gden = scratch + (size_t)p.BH * p.N;
  a.part_S = scratch + dg_f;
  a.part_z = a.part_S + npieces * kD * kD;
  a.seg_chunks = (int)seg_chunks;
  a.nseg = (int)G;
  a.parts = (int)parts;
  a.N = p.N;
  a.eps = p.eps;
  {
    LaunchTimer timer(kKBackward, p.stream);
    if (G > 1) {
      bwd_state_tc<<<dim3((unsigned)((G - 1) * parts), (unsigned)p.BH), kStThreads, StLayout::Bytes, p.stream>>>(a);
      e = cudaGetLastError();
      if (e == cudaSuccess) count_launch();
    }
    if (e == cudaSuccess) {
      bwd_pass1_tc<<<dim3((unsigned)G, (unsigned)p.BH), kP1Threads, P1Layout::Bytes, p.stream>>>(a);
      e = cudaGetLastError();
    }
    if (e == cudaSuccess) {
      count_launch();
      bwd_pass2_tc<<<dim3((unsigned)p.BH, 2), kP2Threads, P2Layout::Bytes, p.stream>>>(a);
      e = cudaGetLastError();
    }
    if (e == cudaSuccess) count_launch();
    timer.done(e);
  }
  const cudaError_t f = cudaFreeAsync(scratch, p.stream);
  return e != cudaSuccess ? e : f;
}

cudaError_t read_and_clear_backward_status(unsigned int *value) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(value, g_bwd_status, sizeof(unsigned int));
  if (e == cudaSuccess && *value) e = cudaMemcpyToSymbol(g_bwd_status, &zero, sizeof(unsigned int));
  return e;
}

}  // namespace la
