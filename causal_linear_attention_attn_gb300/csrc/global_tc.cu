// Global (non-causal) linear attention on the sm_103a tensor cores.
//
// S = sum_j phi(k_j) v_j^T and z = sum_j phi(k_j) over the whole sequence,
// then o_i = phi(q_i)^T S / (phi(q_i)^T z + eps) for every position
// ("Linear Attention Math", "Linear attention by associativity";
// "线性注意力从头到尾讲清楚" §4 and the sketch in §8).  Two kernels:
//
// 1. State build: a cluster of G CTAs per head, each over a contiguous range
//    of tokens.  TMA lands K and V tiles (128-byte swizzle); eight warps
//    apply phi to K in place (bf16), zero the rows past the end and add the
//    rounded values into fp32 column sums (z); one thread issues
//    S += phi(K)^T V (M = N = 128) into an fp32 tensor-memory accumulator.
//    For d = 64 the 128 rows of M are two 128-token sub-tiles side by side:
//    the MMA forms [K_a | K_b]^T [V_a | V_b], whose two diagonal 64x64 blocks
//    are the sub-tiles' contributions (the off-diagonal blocks are unused).
//    The partial states meet through distributed shared memory and the
//    cluster writes S and z.  phi costs one exp per element on the MUFU
//    unit, about as long as the tile's load, so each thread loads all of its
//    chunks before transforming any (the exp latencies overlap).
// 2. Read: persistent CTAs over 128-token tiles.  Eight warps apply phi to
//    the Q tile in place; B = [bf16(S) | hi and lo bf16 parts of z | 0] is built
//    once per head in a K-major layout, so one MMA (M = 128, N = d + 16,
//    K = d) gives every numerator and the denominator; eight warps
//    normalise and stage fp32 rows that TMA stores write out.
//
// Every mbarrier wait is bounded: a wait that runs out raises the CTA's
// abort word and the device status word, and the CTA drains its copies and
// MMAs, frees tensor memory and exits.
#include <cooperative_groups.h>
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace cg = cooperative_groups;

namespace la {

__device__ unsigned int g_global_status;

namespace {
using namespace tc;

constexpr uint32_t kBlk = 16384;           // [128 rows x 128 bytes], 128-byte swizzled
constexpr uint32_t kAbortMisaligned = 2u;  // status bit: shared memory base not 1024-aligned

// phi in place on a tile of 16-byte chunks: thread t of `kThr` takes chunks
// t, t + kThr, ...; all loads are issued before any exp so that their
// latencies overlap.  Chunk c covers row c / 8 of a 128-byte-row tile.
template <int kPer, int kThr, typename F>
__device__ __forceinline__ void phi_chunks(uint8_t *tile, int t, F &&each) {
  uint4 x[kPer];
#pragma unroll
  for (int j = 0; j < kPer; ++j) x[j] = reinterpret_cast<const uint4 *>(tile)[t + kThr * j];
#pragma unroll
  for (int j = 0; j < kPer; ++j) x[j] = each(j, t + kThr * j, x[j]);
#pragma unroll
  for (int j = 0; j < kPer; ++j) reinterpret_cast<uint4 *>(tile)[t + kThr * j] = x[j];
}

// acc[0..7] += the eight bf16 values of y, by packed fp32 adds (acc is 8-byte aligned)
__device__ __forceinline__ void add8_bf16(float *acc, uint4 y) {
  const uint32_t w[4] = {y.x, y.y, y.z, y.w};
  float2 *a2 = reinterpret_cast<float2 *>(acc);
#pragma unroll
  for (int e = 0; e < 4; ++e)
    a2[e] = __fadd2_rn(a2[e], make_float2(__uint_as_float(w[e] << 16), __uint_as_float(w[e] & 0xffff0000u)));
}

// ------------------------------------------------------------------ state build

constexpr int kBuildThreads = 320;  // warp 0 TMA, 1 MMA, 2-9 phi(K) and the epilogue
constexpr int kBuildStages = 6;
constexpr int kBuildPhi = 256;
constexpr uint32_t kBarBuild = 1;   // named barrier of warps 2-9
constexpr uint32_t kHalf = 8192;    // [64 rows x 128 bytes], 128-byte swizzled

// Stages are 64-token (d = 128) or 128-token (d = 64, two 64-token sub-tiles)
// K and V tiles of 16 KB each: a stage is held only for its phi and four
// MMAs, so most of the six stages are loads in flight.  Retention (kRet)
// adds the low bf16 parts of the weighted keys per stage, in four stages.
template <int D, bool kRet = false>
struct BuildLayout {
  static constexpr int kStages = kRet ? 4 : kBuildStages;
  static constexpr uint32_t kStage = 2 * kHalf;  // one K or V stage: 16 KB
  static constexpr uint32_t K = 0;
  static constexpr uint32_t V = K + kStages * kStage;
  static constexpr uint32_t Klo = V + kStages * kStage;  // retention only
  static constexpr int kZ = D == 64 ? 8 : 16;  // column sums per feature-map thread
  static constexpr uint32_t Zred = Klo + (kRet ? kStages * kStage : 0);  // [256 threads][kZ] column sums, then z
  static constexpr uint32_t Bars = Zred + kBuildPhi * kZ * 4 + D * 4;
  static constexpr int kNumBars = 3 * kStages + 2;
  static constexpr uint32_t Misc = Bars + kNumBars * 8;
  static constexpr uint32_t Bytes = Misc + 16;
  // partial state [128 rows][D + 4] fp32, written over the K stages (whole-sequence mode)
  static constexpr int kPStride = D + 4;
  static_assert(kRet || 128 * kPStride * 4 <= kStages * kStage, "partial state fits over the K stages");
};
static_assert(BuildLayout<128>::Bytes <= 232448, "shared memory budget");
static_assert(BuildLayout<128, true>::Bytes <= 232448, "shared memory budget");

struct BuildParams {
  CUtensorMap tk, tv;  // [BH][N][D] bf16, boxes 64 x 64 x 1 (d = 128) or 64 x 128 x 1 (d = 64), 128-byte swizzle
  float *S, *z;        // whole-sequence mode: final state, summed over the cluster
  // Range mode (part_S non-null, d = 128): the first pass of the causal form.  Head h's
  // ranges r = h * ranges_per_head + s (s < ranges_per_head) cover its units
  // [s * range_units, (s + 1) * range_units); all heads' ranges, one after another, form
  // units_total flattened units, split evenly over the CTAs of a 1-D grid.  A CTA's run
  // is at most one range long, so it touches at most two ranges: its pieces 0 and 1 go to
  // part_S[(2 c + k)][D][D] and part_z[(2 c + k)][D] (an empty piece 1 is written as zeros).
  // With pieces_per_cta == 1 the runs divide the ranges evenly and CTA c writes piece c only.
  float *part_S, *part_z;
  long N;
  int units;  // stage units per head: 128 tokens (d = 64) or 64 (d = 128)
  long units_total;
  int range_units, ranges_per_head, pieces_per_cta;
  // Retention (range mode, kRet): key rows of a piece are weighted by gamma^(piece end - 1 - t)
  // with head bh's gamma = 2^log2g[bh % ret_H]; the key sums are not formed.
  int ret_H;
  float log2g[kMaxRetentionHeads];
};

// Walks stage units as (head, unit in head) pairs without per-unit division.
struct UnitWalk {
  int h;
  long u;
  long per_head;
  __device__ void next() {
    if (++u == per_head) {
      u = 0;
      ++h;
    }
  }
};

template <int D, int kMode = kModeElu>
__global__ void __launch_bounds__(kBuildThreads, 1) global_build_tc(const __grid_constant__ BuildParams p) {
  constexpr bool kRet = kMode == kModeRetention;
  using Lay = BuildLayout<D, kRet>;
  constexpr int kBuildStages = Lay::kStages;
  constexpr int kUnit = D == 64 ? 128 : 64;
  constexpr int kPS = Lay::kPStride;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // every CTA sees the same base, so either all return here or none does
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) atomicOr(&g_global_status, kAbortMisaligned);
    return;
  }
  uint8_t *sm = smem_raw;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + Lay::Bars);
  uint64_t *full = bars, *phi_done = bars + kBuildStages, *empty = bars + 2 * kBuildStages,
           *acc_full = bars + 3 * kBuildStages, *drain = acc_full + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + Lay::Misc);
  volatile uint32_t *abort_word = reinterpret_cast<volatile uint32_t *>(sm + Lay::Misc + 4);
  unsigned int *status = &g_global_status;
  float *P = reinterpret_cast<float *>(sm + Lay::K);
  float *zred = reinterpret_cast<float *>(sm + Lay::Zred), *zpart = zred + kBuildPhi * Lay::kZ;

  const bool range_mode = D == 128 && p.part_S != nullptr;
  cg::cluster_group cluster = cg::this_cluster();
  const int G = range_mode ? 1 : (int)cluster.num_blocks(), rank = range_mode ? 0 : (int)cluster.block_rank();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // this CTA's units: nu of them from (h0, uh0); the units from nb on form piece 1
  UnitWalk start;
  int nu, nb;
  if (range_mode) {
    start.per_head = (long)p.ranges_per_head * p.range_units;
    const long f0 = p.units_total * blockIdx.x / gridDim.x, f1 = p.units_total * (blockIdx.x + 1) / gridDim.x;
    nu = (int)(f1 - f0);
    start.h = (int)(f0 / start.per_head);
    start.u = f0 - (long)start.h * start.per_head;
    nb = p.pieces_per_cta == 1 ? nu : (int)min((long)nu, (f0 / p.range_units + 1) * p.range_units - f0);
  } else {
    start.per_head = p.units;
    start.h = blockIdx.y;
    start.u = (long)p.units * rank / G;
    nu = (int)((long)p.units * (rank + 1) / G - start.u);
    nb = nu;
  }
  nu = max(nu, 0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kBuildStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&phi_done[s], kBuildPhi);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(drain, 1);
    *abort_word = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, 256);
  // the kernel queued after this one (the read, or the main causal pass) may start on free SMs
  if (threadIdx.x == 0) pdl_trigger();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem;  // piece k accumulates at columns 128 k

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      prefetch_tmap(&p.tk);
      prefetch_tmap(&p.tv);
      UnitWalk w = start;
      int issued = 0;
      for (int i = 0; i < nu; ++i, w.next()) {
        const int s = i % kBuildStages;
        const uint32_t r = i / kBuildStages;
        if (i >= kBuildStages && !mbar_wait(&empty[s], (r - 1) & 1, abort_word, status)) break;
        const int tok = (int)w.u * kUnit;
        uint8_t *k = sm + Lay::K + s * Lay::kStage, *v = sm + Lay::V + s * Lay::kStage;
        mbar_arrive_expect_tx(&full[s], 2 * Lay::kStage);
        // d = 64: one 128-token box per tensor, whose rows 0-63 and 64-127 are the two 64-token
        // sub-tiles (fewer, larger copies stream faster); d = 128: the two 64-feature halves
        tma_load_3d(k, &p.tk, &full[s], 0, tok, w.h);
        tma_load_3d(v, &p.tv, &full[s], 0, tok, w.h);
        if (D == 128) {
          tma_load_3d(k + kHalf, &p.tk, &full[s], 64, tok, w.h);
          tma_load_3d(v + kHalf, &p.tv, &full[s], 64, tok, w.h);
        }
        issued = i + 1;
      }
      for (int i = max(0, issued - kBuildStages); i < issued; ++i)
        wait_drain(&full[i % kBuildStages], (i / kBuildStages) & 1, status);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t iS = idesc_bf16_f32(128, 128, 1, 1);
      const uint32_t sK = smem_u32(sm + Lay::K), sV = smem_u32(sm + Lay::V), sKlo = smem_u32(sm + Lay::Klo);
      for (int i = 0; i < nu; ++i) {
        const int s = i % kBuildStages;
        if (!mbar_wait(&phi_done[s], (i / kBuildStages) & 1, abort_word, status)) break;
        tc_fence_after();
        const uint32_t k = sK + s * Lay::kStage, v = sV + s * Lay::kStage;
        const uint32_t d = tS + (i >= nb ? 128u : 0u);
        const bool first = i == 0 || i == nb;  // a piece's first unit overwrites its accumulator
#pragma unroll 1
        for (int ks = 0; ks < 4; ++ks) {  // both operands MN-major: 16 tokens per step, 64-wide blocks 8 KB apart
          mma_bf16(d, sw128_desc(k + ks * 2048, kHalf, 1024), sw128_desc(v + ks * 2048, kHalf, 1024), iS,
                   (!first || ks > 0) ? 1u : 0u);
          if (kRet)  // the weighted keys' low parts
            mma_bf16(d, sw128_desc(sKlo + s * Lay::kStage + ks * 2048, kHalf, 1024),
                     sw128_desc(v + ks * 2048, kHalf, 1024), iS, 1u);
        }
        mma_commit(&empty[s]);
      }
      mma_commit(acc_full);
      mma_commit(drain);
      wait_drain(drain, 0, status);
    }
  } else {
    // ---------------- phi(K) in place, column sums, then the partial states ----------------
    const int pt = threadIdx.x - 64;
    // Chunk pt + 256 j sits at position pt & 7 of row (pt >> 3) + 32 j; with the
    // 128-byte swizzle it holds the features 8 g .. 8 g + 7, g = (pt & 7) ^ ((pt >> 3) & 7),
    // of its row (of the 64-feature block j / 2 for d = 128), the same g for every j.
    constexpr int kZ = Lay::kZ;
    float zacc0[kZ], zacc1[kZ];  // per piece (kept in registers: selected by uniform branches)
#pragma unroll
    for (int a = 0; a < kZ; ++a) zacc0[a] = zacc1[a] = 0.f;
    bool failed = false;
    UnitWalk w = start;
    for (int i = 0; i < nu; ++i, w.next()) {
      const int s = i % kBuildStages;
      const bool ok = mbar_wait(&full[s], (i / kBuildStages) & 1, abort_word, status);
      if (bar_or(kBarBuild, kBuildPhi, !ok)) {
        failed = true;
        break;
      }
      uint8_t *k = sm + Lay::K + s * Lay::kStage;
      const long tok0 = w.u * kUnit;
      if constexpr (kRet) {
        // retention: row t of the unit weighted by gamma^(tokens from t to the piece end - 1), as a
        // bf16 pair: the high parts in place, the low parts in this stage's Klo tile
        const float lg = p.log2g[w.h % max(p.ret_H, 1)];
        const float to_end = (float)(kUnit * ((i < nb ? nb : nu) - i));
        uint4 *kt = reinterpret_cast<uint4 *>(k), *lt = reinterpret_cast<uint4 *>(sm + Lay::Klo + s * Lay::kStage);
        uint4 x[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) x[j] = kt[pt + kBuildPhi * j];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int ch = pt + kBuildPhi * j, row = (ch >> 3) & 63;  // the unit's token row
          uint4 hi = make_uint4(0u, 0u, 0u, 0u), lo = hi;          // rows past the end add nothing
          if (tok0 + row < p.N) split8(x[j], exp2f((to_end - 1.f - (float)row) * lg), hi, lo);
          kt[ch] = hi;
          lt[ch] = lo;
        }
      } else {
        // phi in place; the rounded values also go into the column sums of this unit's piece
        auto phi_sum = [&](float *za) {
          phi_chunks<4, kBuildPhi>(k, pt, [&](int j, int ch, uint4 x) {
            const int row = ch >> 3;  // 0..127 over the two blocks
            const long tok = tok0 + (D == 64 ? row : (row & 63));
            // rows past the end add nothing; given features (identity mode) pass unchanged
            const uint4 y = tok >= p.N ? make_uint4(0u, 0u, 0u, 0u) : kMode == kModeIdentity ? x : phi8(x);
            add8_bf16(za + (D == 64 ? 0 : 8 * (j >> 1)), y);
            return y;
          });
        };
        if (i < nb)
          phi_sum(zacc0);
        else
          phi_sum(zacc1);
      }
      fence_async_smem();
      mbar_arrive(&phi_done[s]);
    }
    bool ok = !failed && mbar_wait(acc_full, 0, abort_word, status);
    ok = !bar_or(kBarBuild, kBuildPhi, !ok);
    const int quarter = warp & 3, half = (warp - 2) >> 2, row = quarter * 32 + lane;
    const uint32_t lanes = (uint32_t)(quarter * 32) << 16;
    const int npieces = range_mode ? p.pieces_per_cta : 1;
#pragma unroll
    for (int piece = 0; piece < 2; ++piece) {
      if (piece >= npieces) break;
      const bool filled = ok && (piece == 0 ? min(nu, nb) > 0 : nu > nb);
      const float *zp = piece == 0 ? zacc0 : zacc1;
      // column sums: feature f = 64 b + 8 g + e is held, as entry 8 b + e (d = 128) or e,
      // by the 32 threads 8 m + (g ^ (m & 7)), m = 0..31
#pragma unroll
      for (int a = 0; a < kZ; ++a) zred[pt * kZ + a] = zp[a];
      named_bar(kBarBuild, kBuildPhi);
      if (pt < D) {
        const int b = pt >> 6, g = (pt >> 3) & 7, e = pt & 7;
        float zs = 0.f;
#pragma unroll 8
        for (int m = 0; m < 32; ++m) zs += zred[(8 * m + (g ^ (m & 7))) * kZ + (D == 64 ? e : 8 * b + e)];
        zs = filled ? zs : 0.f;
        if (range_mode)
          p.part_z[((long)p.pieces_per_cta * blockIdx.x + piece) * D + pt] = zs;
        else
          zpart[pt] = zs;
      }
      named_bar(kBarBuild, kBuildPhi);  // zred is free for the next piece
      // range mode: row `row` of the piece goes straight to global memory; otherwise to shared memory
      const long slot = (long)p.pieces_per_cta * blockIdx.x + piece;
      float *prow = range_mode ? p.part_S + (slot * D + row) * D : P + row * kPS;
      if (filled) {
        tc_fence_after();
        uint32_t v[32];
        constexpr int kParts = D == 64 ? 1 : 2;
#pragma unroll
        for (int c = 0; c < kParts; ++c) {
          // d = 64: rows 0-63 hold K_a^T V_a in columns 0-63, rows 64-127 K_b^T V_b in columns 64-127
          const int src = D == 64 ? (row < 64 ? 0 : 64) + 32 * half : 64 * half + 32 * c;
          const int dst = D == 64 ? 32 * half : 64 * half + 32 * c;
          tmem_ld32(tS + 128 * piece + lanes + src, v);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *reinterpret_cast<float4 *>(prow + dst + 4 * q) =
                make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                            __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
        }
      } else if (range_mode) {
        // an empty piece reads as zeros: coalesced 16-byte stores over the whole [D][D] piece
        float4 *z4 = reinterpret_cast<float4 *>(p.part_S + slot * D * D);
        for (int e = pt; e < D * D / 4; e += kBuildPhi) z4[e] = make_float4(0.f, 0.f, 0.f, 0.f);
      } else {
        const int wd = D == 64 ? 32 : 64;
        for (int c = 0; c < wd; ++c) prow[wd * half + c] = 0.f;
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  if (range_mode) {
    // pieces and their key sums were written above; the barrier keeps tensor
    // memory allocated until every read of it is done
    __syncthreads();
  } else {
    const int bh = blockIdx.y;
    cluster.sync();  // every partial state of the cluster is in shared memory
    // this CTA sums rows [r0, r0 + D/G) of S (and those entries of z) over the cluster
    const int rows = D / G, r0 = rank * rows;
    for (int e = threadIdx.x; e < rows * (D + 1); e += kBuildThreads) {
      const int i = r0 + e / (D + 1), j = e % (D + 1);
      float acc = 0.f;
      for (int c = 0; c < G; ++c) {
        if (j == D) {
          acc += cluster.map_shared_rank(zpart, c)[i];
          continue;
        }
        const float *Pc = cluster.map_shared_rank(P, c);
        acc += Pc[i * kPS + j];
        if (D == 64) acc += Pc[(64 + i) * kPS + j];
      }
      if (j < D)
        p.S[((long)bh * D + i) * D + j] = acc;
      else
        p.z[(long)bh * D + i] = acc;
    }
    cluster.sync();  // remote reads are done before any CTA of the cluster exits
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// ------------------------------------------------------------------ read

constexpr int kReadThreads = 576;  // warp 0 TMA, 1 MMA, 2-9 phi(Q) and B, 10-17 epilogue
constexpr int kReadPhi = 256, kReadEpi = 256;
constexpr uint32_t kBarEpi = 1, kBarPhi = 2;

template <int D>
struct ReadLayout {
  static constexpr int kStages = D == 64 ? 6 : 2;  // Q tiles in flight
  static constexpr int NB = D + 16;             // B rows: d columns of S, z hi, z lo, zero padding
  static constexpr uint32_t kQ = D * 2 * 128;   // one Q tile (D/64 swizzled 16 KB blocks)
  static constexpr uint32_t kAtomB = NB * 128;  // one 64-wide K atom of B
  static constexpr uint32_t kB = (D / 64) * kAtomB;
  static constexpr int kOutBufs = D == 64 ? 2 : 1;
  static constexpr uint32_t kOut = D * 4 * 128;  // one fp32 tile: D/32 boxes of [128 x 32]
  static constexpr uint32_t Q = 0;
  static constexpr uint32_t B = Q + kStages * kQ;  // two buffers (heads alternate)
  static constexpr uint32_t O = B + 2 * kB;
  static constexpr uint32_t Bars = O + kOutBufs * kOut;
  static constexpr int kNumBars = 3 * kStages + 8;
  static constexpr uint32_t Misc = Bars + kNumBars * 8;
  static constexpr uint32_t Bytes = Misc + 16;
  static constexpr uint32_t kAccCols = D == 64 ? 128 : 256;  // column distance of the two accumulators
  static constexpr uint32_t TmemCols = 2 * kAccCols;
  static_assert(kAtomB % 1024 == 0 && kB % 1024 == 0, "B atoms stay 1024-aligned");
};
static_assert(ReadLayout<128>::Bytes <= 232448, "shared memory budget");

struct ReadParams {
  CUtensorMap tq;  // [BH][N][D] bf16, box 64 x 128 x 1, 128-byte swizzle
  CUtensorMap to;  // [BH][N][D] fp32, box 32 x 128 x 1, 128-byte swizzle
  const float *S, *z;
  long N;
  int tiles_per_head;
  long total_tiles;
  float eps;
};

// Walks a CTA's contiguous run of 128-token tiles as (head, tile in head)
// pairs: one division at the start, none per tile (64-bit division is a long
// software sequence and sat on every role's per-tile path).
struct TileWalk {
  int bh, t, tph;
  __device__ TileWalk(long first, int tiles_per_head)
      : bh((int)(first / tiles_per_head)), t((int)(first % tiles_per_head)), tph(tiles_per_head) {}
  __device__ void next() {
    if (++t == tph) {
      t = 0;
      ++bh;
    }
  }
  __device__ bool last_of_head() const { return t == tph - 1; }
};

__device__ __forceinline__ void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }

// B for one head, K-major and 128-byte swizzled: row n < D holds column n of
// S over the D key features (bf16), rows D and D+1 the hi and lo bf16 parts
// of z, the rest zeros.  256 threads; consecutive threads take consecutive
// rows, so the reads of S are coalesced and the swizzled stores conflict-free.
template <int D>
__device__ __forceinline__ void build_b(uint8_t *B, const float *__restrict__ S, const float *__restrict__ z,
                                        int t) {
  using Lay = ReadLayout<D>;
  constexpr int NB = Lay::NB, kChunks = D / 8;  // 16-byte chunks per row
  for (int e = t; e < kChunks * NB; e += kReadPhi) {
    const int n = e % NB, c = e / NB;
    uint32_t w[4];
    if (n < D) {
#pragma unroll
      for (int j = 0; j < 4; ++j) w[j] = pack_bf16(S[(8 * c + 2 * j) * D + n], S[(8 * c + 2 * j + 1) * D + n]);
    } else if (n < D + 2) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float a = z[8 * c + 2 * j], b = z[8 * c + 2 * j + 1];
        const float ah = __bfloat162float(__float2bfloat16_rn(a)), bh = __bfloat162float(__float2bfloat16_rn(b));
        w[j] = n == D ? pack_bf16(ah, bh) : pack_bf16(a - ah, b - bh);
      }
    } else {
      w[0] = w[1] = w[2] = w[3] = 0u;
    }
    const int atom = c >> 3, cc = c & 7;
    *reinterpret_cast<uint4 *>(B + atom * Lay::kAtomB + n * 128 + ((cc ^ (n & 7)) << 4)) =
        make_uint4(w[0], w[1], w[2], w[3]);
  }
}

template <int D>
__global__ void __launch_bounds__(kReadThreads, 1) global_read_tc(const __grid_constant__ ReadParams p) {
  using Lay = ReadLayout<D>;
  constexpr int NB = Lay::NB;
  constexpr int kStages = Lay::kStages;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) atomicOr(&g_global_status, kAbortMisaligned);
    return;
  }
  uint8_t *sm = smem_raw;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + Lay::Bars);
  uint64_t *full = bars, *phi_done = bars + kStages, *q_empty = bars + 2 * kStages,
           *acc_full = bars + 3 * kStages,  // [2]
      *acc_empty = acc_full + 2,                // [2]
      *b_free = acc_full + 4,                   // [2]
      *drain = acc_full + 6;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + Lay::Misc);
  volatile uint32_t *abort_word = reinterpret_cast<volatile uint32_t *>(sm + Lay::Misc + 4);
  unsigned int *status = &g_global_status;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long t_lo = p.total_tiles * blockIdx.x / gridDim.x;
  const long t_hi = p.total_tiles * (blockIdx.x + 1) / gridDim.x;
  const int n = (int)(t_hi - t_lo);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&phi_done[s], kReadPhi);
      mbar_init(&q_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], kReadEpi / 32);
      mbar_init(&b_free[b], 1);
    }
    mbar_init(drain, 1);
    *abort_word = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, Lay::TmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      prefetch_tmap(&p.tq);
      TileWalk w(t_lo, p.tiles_per_head);
      int issued = 0;
      for (int i = 0; i < n; ++i) {
        const int s = i % kStages;
        const uint32_t r = i / kStages;
        if (i >= kStages && !mbar_wait(&q_empty[s], (r - 1) & 1, abort_word, status)) break;
        const int bh = w.bh, tok = w.t * 128;
        w.next();
        uint8_t *q = sm + Lay::Q + s * Lay::kQ;
        mbar_arrive_expect_tx(&full[s], Lay::kQ);
#pragma unroll
        for (int b = 0; b < D / 64; ++b) tma_load_3d(q + b * kBlk, &p.tq, &full[s], 64 * b, tok, bh);
        issued = i + 1;
      }
      for (int i = max(0, issued - kStages); i < issued; ++i)
        wait_drain(&full[i % kStages], (i / kStages) & 1, status);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t iR = idesc_bf16_f32(128, NB, 0, 0);
      const uint32_t sQ = smem_u32(sm + Lay::Q), sB = smem_u32(sm + Lay::B);
      int hl = 0;  // local head index: B buffer hl & 1
      TileWalk w(t_lo, p.tiles_per_head);
      for (int i = 0; i < n; ++i, w.next()) {
        const int s = i % kStages, buf = i & 1;
        if (i > 0 && w.t == 0) ++hl;
        if (!mbar_wait(&phi_done[s], (i / kStages) & 1, abort_word, status)) break;
        if (i >= 2 && !mbar_wait(&acc_empty[buf], ((i >> 1) - 1) & 1, abort_word, status)) break;
        tc_fence_after();
        const uint32_t d = tmem + buf * Lay::kAccCols, q = sQ + s * Lay::kQ, b = sB + (hl & 1) * Lay::kB;
#pragma unroll 1
        for (int ks = 0; ks < D / 16; ++ks)
          mma_bf16(d, sw128_desc(q + (ks >> 2) * kBlk + (ks & 3) * 32, 16, 1024),
                   sw128_desc(b + (ks >> 2) * Lay::kAtomB + (ks & 3) * 32, 16, 1024), iR, ks > 0 ? 1u : 0u);
        mma_commit(&q_empty[s]);
        mma_commit(&acc_full[buf]);
        // the last tile of a head frees its B buffer once these MMAs complete
        if (i == n - 1 || w.last_of_head()) mma_commit(&b_free[hl & 1]);
      }
      mma_commit(drain);
      wait_drain(drain, 0, status);
    }
  } else if (warp < 10) {
    // ---------------- phi(Q) in place, and B per head ----------------
    const int pt = threadIdx.x - 64;
    int hl = -1;
    TileWalk w(t_lo, p.tiles_per_head);
    for (int i = 0; i < n; ++i, w.next()) {
      const int s = i % kStages;
      const long bh = w.bh;
      if (i == 0 || w.t == 0) {
        ++hl;
        // B buffer hl & 1 last served head hl - 2
        const bool ok = hl < 2 || mbar_wait(&b_free[hl & 1], ((hl >> 1) - 1) & 1, abort_word, status);
        if (bar_or(kBarPhi, kReadPhi, !ok)) break;
        if (hl == 0) pdl_wait();  // S and z come from the state build: complete and visible
        build_b<D>(sm + Lay::B + (hl & 1) * Lay::kB, p.S + bh * D * D, p.z + bh * D, pt);
      }
      const bool ok = mbar_wait(&full[s], (i / kStages) & 1, abort_word, status);
      if (bar_or(kBarPhi, kReadPhi, !ok)) break;
      phi_chunks<(int)(Lay::kQ / 16) / kReadPhi, kReadPhi>(sm + Lay::Q + s * Lay::kQ, pt,
                                                          [](int, int, uint4 x) { return phi8(x); });
      fence_async_smem();
      mbar_arrive(&phi_done[s]);
    }
  } else {
    // ---------------- epilogue: normalise, stage, TMA store ----------------
    const int et = threadIdx.x - 320;  // 0..255
    const int quarter = warp & 3, half = (warp - 10) >> 2, row = quarter * 32 + lane;
    const uint32_t lanes = (uint32_t)(quarter * 32) << 16;
    TileWalk w(t_lo, p.tiles_per_head);
    for (int i = 0; i < n; ++i, w.next()) {
      const int buf = i & 1, ob = i % Lay::kOutBufs;
      const int bh = w.bh, tok = w.t * 128;
      const bool ok = mbar_wait(&acc_full[buf], (i >> 1) & 1, abort_word, status);
      if (bar_or(kBarEpi, kReadEpi, !ok)) break;
      tc_fence_after();
      const uint32_t ta = tmem + buf * Lay::kAccCols + lanes;
      const float den = __uint_as_float(tmem_ld1(ta + D)) + __uint_as_float(tmem_ld1(ta + D + 1));
      const float inv = 1.f / (den + p.eps);
      constexpr int kParts = D / 64;  // 32-column loads per thread
      uint32_t v[kParts][32];
#pragma unroll
      for (int c = 0; c < kParts; ++c) tmem_ld32(ta + (D / 2) * half + 32 * c, v[c]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
      // the staging buffer is free once the store issued from it kOutBufs tiles ago has read it
      if (et == 0) {
        if (Lay::kOutBufs == 2)
          bulk_wait_read_1();
        else
          bulk_wait_read();
      }
      named_bar(kBarEpi, kReadEpi);
      uint8_t *stage = sm + Lay::O + ob * Lay::kOut;
#pragma unroll
      for (int c = 0; c < kParts; ++c) {
        uint8_t *box = stage + ((D / 64) * half + c) * kBlk;  // box b holds columns [32b, 32b + 32)
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) {
          const float2 a = __fmul2_rn(make_float2(__uint_as_float(v[c][4 * q4]), __uint_as_float(v[c][4 * q4 + 1])),
                                      make_float2(inv, inv));
          const float2 b = __fmul2_rn(make_float2(__uint_as_float(v[c][4 * q4 + 2]),
                                                  __uint_as_float(v[c][4 * q4 + 3])),
                                      make_float2(inv, inv));
          *reinterpret_cast<float4 *>(box + sw128_offset_f32(row, 4 * q4)) = make_float4(a.x, a.y, b.x, b.y);
        }
      }
      fence_async_smem();
      named_bar(kBarEpi, kReadEpi);
      if (et == 0) {
#pragma unroll
        for (int b = 0; b < D / 32; ++b) tma_store_3d(&p.to, stage + b * kBlk, 32 * b, tok, bh);
        bulk_commit();
      }
    }
    if (et == 0) bulk_wait_all();  // output stores complete before the CTA exits
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Lay::TmemCols);
  }
}

// ------------------------------------------------------------------ one pass (d = 64, a CTA per head)

// When the heads alone fill the SMs, one CTA per head builds S and z and then
// reads every query of the same head: no kernel boundary and no grid-wide
// wait lie between the two halves, and the head's first query tiles load
// while its last key and value units are still being summed.
//
// Build: 128-token K | V units in a six-slot ring, phi(K) by sixteen warps,
// S += phi(K)^T V with the two 64-token sub-tiles side by side (as in the
// state build).  Hand-over: the column sums and S (the two diagonal blocks of
// the accumulator) go to global memory and, as B = [bf16(S) | z hi | z lo | 0],
// to shared memory.  Read: 128-token Q tiles in eight 16 KB stages over the
// first four ring slots, phi(Q) by eight warps, one M = 128, N = 80, K = 64
// MMA a tile into one of two accumulators, eight epilogue warps normalising
// into two fp32 staging tiles over the last two ring slots.
constexpr int kFusedThreads = 576;  // warp 0 TMA, 1 MMA, 2-17 phi(K); then 2-9 phi(Q), 10-17 epilogue
constexpr int kFusedA = 512, kFusedPhi = 256, kFusedEpi = 256;
constexpr uint32_t kBarFusedA = 1, kBarFusedEpi = 2;

struct FusedLayout {
  static constexpr int kSlots = 6;                  // K | V units
  static constexpr uint32_t kSlot = 2 * kBlk;       // 32 KB: K then V, [128 tokens x 64] each
  static constexpr int kQStages = 8;                // Q tiles of 16 KB over slots 0-3
  static constexpr int NB = 80;                     // B rows: 64 columns of S, z hi, z lo, zeros
  static constexpr uint32_t Out = 4 * kSlot;        // two fp32 output tiles of 32 KB over slots 4-5
  static constexpr uint32_t Zred = Out;             // hand-over: [512 threads][8] column sums
  static constexpr uint32_t Pst = Zred + kFusedA * 8 * 4;  // hand-over: accumulator rows [128][68] fp32
  static constexpr int kPStride = 68;
  static constexpr uint32_t B = kSlots * kSlot;
  static constexpr uint32_t Zs = B + NB * 128;
  static constexpr uint32_t Bars = Zs + 64 * 4;
  static constexpr int kNumBars = 3 * kSlots + 2 + 3 * kQStages + 5;
  static constexpr uint32_t Misc = Bars + kNumBars * 8;
  static constexpr uint32_t Bytes = Misc + 16;
  static_assert(Pst + 128 * kPStride * 4 <= B, "hand-over staging fits over slots 4-5");
  static_assert(kQStages * kBlk <= Out, "Q stages fit over slots 0-3");
  static_assert(B % 1024 == 0, "B stays 1024-aligned");
};
static_assert(FusedLayout::Bytes <= 232448, "shared memory budget");

struct FusedParams {
  CUtensorMap tk, tv, tq;  // [BH][N][64] bf16, box 64 x 128 x 1, 128-byte swizzle
  CUtensorMap to;          // [BH][N][64] fp32, box 32 x 128 x 1, 128-byte swizzle
  float *S, *z;
  long N;
  float eps;
};

__global__ void __launch_bounds__(kFusedThreads, 1) global_fused_tc(const __grid_constant__ FusedParams p) {
  using Lay = FusedLayout;
  constexpr int kSA = Lay::kSlots, kSB = Lay::kQStages, NB = Lay::NB, kPS = Lay::kPStride;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) atomicOr(&g_global_status, kAbortMisaligned);
    return;
  }
  uint8_t *sm = smem_raw;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + Lay::Bars);
  // build: unit landed, phi applied, slot free; S complete; B written
  uint64_t *full = bars, *phi_done = bars + kSA, *empty = bars + 2 * kSA, *s_full = bars + 3 * kSA,
           *b_ready = s_full + 1;
  // read: Q landed, phi applied, Q stage free; accumulator full / read out (two of each)
  uint64_t *full_q = b_ready + 1, *phi_q = full_q + kSB, *q_empty = phi_q + kSB, *acc_full = q_empty + kSB,
           *acc_empty = acc_full + 2, *drain = acc_empty + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + Lay::Misc);
  volatile uint32_t *abort_word = reinterpret_cast<volatile uint32_t *>(sm + Lay::Misc + 4);
  unsigned int *status = &g_global_status;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.x;
  const int n = (int)((p.N + 127) / 128);  // build units = read tiles

  if (threadIdx.x == 0) {
    for (int s = 0; s < kSA; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&phi_done[s], kFusedA);
      mbar_init(&empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(b_ready, kFusedA);
    for (int t = 0; t < kSB; ++t) {
      mbar_init(&full_q[t], 1);
      mbar_init(&phi_q[t], kFusedPhi);
      mbar_init(&q_empty[t], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], kFusedEpi / 32);
    }
    mbar_init(drain, 1);
    *abort_word = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;  // build: S in columns 0-127; read: accumulators at 0 and 128

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      prefetch_tmap(&p.tk);
      prefetch_tmap(&p.tv);
      prefetch_tmap(&p.tq);
      int issued_a = 0, issued_b = 0;
      for (int i = 0; i < n; ++i) {
        const int s = i % kSA;
        if (i >= kSA && !mbar_wait(&empty[s], (uint32_t)(i / kSA - 1) & 1, abort_word, status)) break;
        uint8_t *u = sm + s * Lay::kSlot;
        mbar_arrive_expect_tx(&full[s], Lay::kSlot);
        tma_load_3d(u, &p.tk, &full[s], 0, i * 128, bh);
        tma_load_3d(u + kBlk, &p.tv, &full[s], 0, i * 128, bh);
        issued_a = i + 1;
      }
      for (int j = 0; issued_a == n && j < n; ++j) {
        const int t = j % kSB;
        if (j < kSB) {
          // stage t lies in slot t / 2: it is free once that slot's last unit has been summed
          const int s = t >> 1;
          if (s < n) {
            const int last = s + kSA * ((n - 1 - s) / kSA);
            if (!mbar_wait(&empty[s], (uint32_t)(last / kSA) & 1, abort_word, status)) break;
          }
        } else if (!mbar_wait(&q_empty[t], (uint32_t)(j / kSB - 1) & 1, abort_word, status)) {
          break;
        }
        mbar_arrive_expect_tx(&full_q[t], kBlk);
        tma_load_3d(sm + t * kBlk, &p.tq, &full_q[t], 0, j * 128, bh);
        issued_b = j + 1;
      }
      // every issued copy must land before shared memory is released
      for (int i = max(0, issued_a - kSA); i < issued_a; ++i)
        wait_drain(&full[i % kSA], (uint32_t)(i / kSA) & 1, status);
      for (int j = max(0, issued_b - kSB); j < issued_b; ++j)
        wait_drain(&full_q[j % kSB], (uint32_t)(j / kSB) & 1, status);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t iS = idesc_bf16_f32(128, 128, 1, 1);
      constexpr uint32_t iR = idesc_bf16_f32(128, NB, 0, 0);
      const uint32_t sR = smem_u32(sm), sB = smem_u32(sm + Lay::B);
      int i = 0;
      for (; i < n; ++i) {
        const int s = i % kSA;
        if (!mbar_wait(&phi_done[s], (uint32_t)(i / kSA) & 1, abort_word, status)) break;
        tc_fence_after();
        const uint32_t k = sR + s * Lay::kSlot, v = k + kBlk;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)  // both operands MN-major: 16 tokens per step, 64-wide blocks 8 KB apart
          mma_bf16(tmem, sw128_desc(k + ks * 2048, kHalf, 1024), sw128_desc(v + ks * 2048, kHalf, 1024), iS,
                   (i > 0 || ks > 0) ? 1u : 0u);
        mma_commit(&empty[s]);
      }
      if (i == n) mma_commit(s_full);
      if (i == n && mbar_wait(b_ready, 0, abort_word, status)) {
        for (int j = 0; j < n; ++j) {
          const int t = j % kSB, buf = j & 1;
          if (!mbar_wait(&phi_q[t], (uint32_t)(j / kSB) & 1, abort_word, status)) break;
          if (j >= 2 && !mbar_wait(&acc_empty[buf], (uint32_t)((j >> 1) - 1) & 1, abort_word, status)) break;
          tc_fence_after();
          const uint32_t d = tmem + 128u * buf, q = sR + t * kBlk;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_bf16(d, sw128_desc(q + ks * 32, 16, 1024), sw128_desc(sB + ks * 32, 16, 1024), iR,
                     ks > 0 ? 1u : 0u);
          mma_commit(&q_empty[t]);
          mma_commit(&acc_full[buf]);
        }
      }
      mma_commit(drain);
      wait_drain(drain, 0, status);
    }
  } else {
    // ---------------- phi(K) in place and column sums (warps 2-17) ----------------
    // Chunk pt + 512 j sits at position pt & 7 of row (pt >> 3) + 64 j and holds the
    // features 8 g .. 8 g + 7, g = (pt & 7) ^ ((pt >> 3) & 7), the same g for both j.
    const int pt = threadIdx.x - 64;  // 0..511
    float za[8];
#pragma unroll
    for (int a = 0; a < 8; ++a) za[a] = 0.f;
    bool failed = false;
    for (int i = 0; i < n; ++i) {
      const int s = i % kSA;
      if (!mbar_wait(&full[s], (uint32_t)(i / kSA) & 1, abort_word, status)) {
        failed = true;
        break;
      }
      const long tok0 = (long)i * 128;
      phi_chunks<2, kFusedA>(sm + s * Lay::kSlot, pt, [&](int, int ch, uint4 x) {
        // rows past the end add nothing
        const uint4 y = tok0 + (ch >> 3) >= p.N ? make_uint4(0u, 0u, 0u, 0u) : phi8(x);
        add8_bf16(za, y);
        return y;
      });
      fence_async_smem();
      mbar_arrive(&phi_done[s]);
    }
    bool ok = !failed && mbar_wait(s_full, 0, abort_word, status) && *abort_word == 0;
    ok = !bar_or(kBarFusedA, kFusedA, !ok);
    // ---------------- hand-over: S and z out, B in ----------------
    if (ok) {
      float *zred = reinterpret_cast<float *>(sm + Lay::Zred), *P = reinterpret_cast<float *>(sm + Lay::Pst);
      float *zs = reinterpret_cast<float *>(sm + Lay::Zs);
#pragma unroll
      for (int a = 0; a < 8; ++a) zred[pt * 8 + a] = za[a];
      tc_fence_after();
      // rows 0-63 hold K_a^T V_a in columns 0-63, rows 64-127 K_b^T V_b in columns 64-127;
      // the four warps of a lane quarter take 16 columns each
      const int quarter = warp & 3, part = (warp - 2) >> 2, row = quarter * 32 + lane;
      uint32_t r[16];
      tmem_ld16(tmem + ((uint32_t)(quarter * 32) << 16) + (row < 64 ? 0u : 64u) + 16u * part, r);
      float *prow = P + row * kPS + 16 * part;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4)
        *reinterpret_cast<float4 *>(prow + 4 * q4) =
            make_float4(__uint_as_float(r[4 * q4]), __uint_as_float(r[4 * q4 + 1]), __uint_as_float(r[4 * q4 + 2]),
                        __uint_as_float(r[4 * q4 + 3]));
      named_bar(kBarFusedA, kFusedA);
      if (pt < 64) {
        const int g = pt >> 3, e = pt & 7;
        float zsum = 0.f;
#pragma unroll 8
        for (int m = 0; m < 64; ++m) zsum += zred[(8 * m + (g ^ (m & 7))) * 8 + e];
        zs[pt] = zsum;
        p.z[(long)bh * 64 + pt] = zsum;
      }
      named_bar(kBarFusedA, kFusedA);
      // B, K-major and 128-byte swizzled: row nn < 64 holds column nn of S over the 64 key
      // features, rows 64 and 65 the hi and lo bf16 parts of z, the rest zeros
      uint8_t *B = sm + Lay::B;
      float *Sg = p.S + (long)bh * 64 * 64;
      for (int e = pt; e < 8 * NB; e += kFusedA) {
        const int nn = e % NB, c = e / NB;
        uint32_t w[4];
        if (nn < 64) {
          float sv[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            sv[j] = P[(8 * c + j) * kPS + nn] + P[(64 + 8 * c + j) * kPS + nn];
            Sg[(8 * c + j) * 64 + nn] = sv[j];
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) w[j] = pack_bf16(sv[2 * j], sv[2 * j + 1]);
        } else if (nn < 66) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float a = zs[8 * c + 2 * j], b = zs[8 * c + 2 * j + 1];
            const float ah = __bfloat162float(__float2bfloat16_rn(a)), bh2 = __bfloat162float(__float2bfloat16_rn(b));
            w[j] = nn == 64 ? pack_bf16(ah, bh2) : pack_bf16(a - ah, b - bh2);
          }
        } else {
          w[0] = w[1] = w[2] = w[3] = 0u;
        }
        *reinterpret_cast<uint4 *>(B + nn * 128 + ((c ^ (nn & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
      }
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(b_ready);
    }

    if (warp < 10) {
      // ---------------- phi(Q) in place ----------------
      for (int j = 0; ok && j < n; ++j) {
        const int t = j % kSB;
        if (!mbar_wait(&full_q[t], (uint32_t)(j / kSB) & 1, abort_word, status)) break;
        phi_chunks<4, kFusedPhi>(sm + t * kBlk, pt, [](int, int, uint4 x) { return phi8(x); });
        fence_async_smem();
        mbar_arrive(&phi_q[t]);
      }
    } else {
      // ---------------- epilogue: normalise, stage, TMA store ----------------
      const int et = threadIdx.x - 320;  // 0..255
      const int quarter = warp & 3, half = (warp - 10) >> 2, row = quarter * 32 + lane;
      const uint32_t lanes = (uint32_t)(quarter * 32) << 16;
      for (int j = 0; ok && j < n; ++j) {
        const int buf = j & 1;
        const bool w = mbar_wait(&acc_full[buf], (uint32_t)(j >> 1) & 1, abort_word, status);
        if (bar_or(kBarFusedEpi, kFusedEpi, !w)) break;
        tc_fence_after();
        const uint32_t ta = tmem + 128u * buf + lanes;
        const float den = __uint_as_float(tmem_ld1(ta + 64)) + __uint_as_float(tmem_ld1(ta + 65));
        const float inv = 1.f / (den + p.eps);
        uint32_t v[32];
        tmem_ld32(ta + 32 * half, v);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[buf]);
        // the staging tile is free once the store issued from it two tiles ago has read it
        if (et == 0) bulk_wait_read_1();
        named_bar(kBarFusedEpi, kFusedEpi);
        uint8_t *stage = sm + Lay::Out + buf * (2 * kBlk);
        uint8_t *box = stage + half * kBlk;  // box b holds columns [32 b, 32 b + 32)
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) {
          const float2 a = __fmul2_rn(make_float2(__uint_as_float(v[4 * q4]), __uint_as_float(v[4 * q4 + 1])),
                                      make_float2(inv, inv));
          const float2 b = __fmul2_rn(make_float2(__uint_as_float(v[4 * q4 + 2]), __uint_as_float(v[4 * q4 + 3])),
                                      make_float2(inv, inv));
          *reinterpret_cast<float4 *>(box + sw128_offset_f32(row, 4 * q4)) = make_float4(a.x, a.y, b.x, b.y);
        }
        fence_async_smem();
        named_bar(kBarFusedEpi, kFusedEpi);
        if (et == 0) {
          tma_store_3d(&p.to, stage, 0, j * 128, bh);
          tma_store_3d(&p.to, stage + kBlk, 32, j * 128, bh);
          bulk_commit();
        }
      }
      if (et == 0) bulk_wait_all();  // output stores complete before the CTA exits
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// ------------------------------------------------------------------ host

bool make_map(CUtensorMap *m, CUtensorMapDataType dt, uint32_t elem, const void *base, long BH, long N, int D,
              uint32_t box_x, uint32_t box_rows) {
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)D * elem, (cuuint64_t)N * D * elem};
  cuuint32_t box[3] = {box_x, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, dt, 3, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The one-pass form for d = 64: a CTA per head.
cudaError_t launch_fused(const Problem &p) {
  FusedParams fp;
  if (!make_map(&fp.tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.k, p.BH, p.N, 64, 64, 128) ||
      !make_map(&fp.tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.v, p.BH, p.N, 64, 64, 128) ||
      !make_map(&fp.tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.q, p.BH, p.N, 64, 64, 128) ||
      !make_map(&fp.to, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p.out, p.BH, p.N, 64, 32, 128))
    return cudaErrorInvalidValue;
  fp.S = p.S;
  fp.z = p.z;
  fp.N = p.N;
  fp.eps = p.eps;
  cudaError_t e = ensure_smem_optin((const void *)global_fused_tc, (int)FusedLayout::Bytes);
  if (e != cudaSuccess) return e;
  LaunchTimer timer(kKGlobalFused, p.stream);
  global_fused_tc<<<(unsigned)p.BH, kFusedThreads, FusedLayout::Bytes, p.stream>>>(fp);
  e = cudaGetLastError();
  timer.done(e);
  if (e == cudaSuccess) count_launch();
  return e;
}

template <int D, int kMode = kModeElu>
cudaError_t build_smem() {
  return ensure_smem_optin((const void *)global_build_tc<D, kMode>, (int)BuildLayout<D, kMode == kModeRetention>::Bytes);
}

template <int D>
cudaError_t launch_t(const Problem &p) {
  const DeviceInfo &di = device_info(-1);
  const long sms = std::max(1, di.sm_count);
  BuildParams bp;
  ReadParams rp;
  // build boxes: 64 features x 64 tokens (d = 128, two per tile) or 64 x 128 (d = 64, one per tile)
  const uint32_t build_rows = D == 64 ? 128 : 64;
  if (!make_map(&bp.tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.k, p.BH, p.N, D, 64, build_rows) ||
      !make_map(&bp.tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.v, p.BH, p.N, D, 64, build_rows) ||
      !make_map(&rp.tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.q, p.BH, p.N, D, 64, 128) ||
      !make_map(&rp.to, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p.out, p.BH, p.N, D, 32, 128))
    return cudaErrorInvalidValue;
  constexpr int kUnit = D == 64 ? 128 : 64;
  bp.S = p.S;
  bp.z = p.z;
  bp.part_S = bp.part_z = nullptr;
  bp.N = p.N;
  bp.units = (int)((p.N + kUnit - 1) / kUnit);
  bp.units_total = 0;
  bp.range_units = bp.ranges_per_head = bp.pieces_per_cta = 0;
  bp.ret_H = 0;
  // cluster size: a power of two <= 8 so that the build covers the SMs about once, >= 8 units a CTA
  int G = 1;
  while (G < 8 && p.BH * (2 * G) <= sms && bp.units / (2 * G) >= 8) G *= 2;
  // a CTA per head covers at least 80 % of the SMs: build and read in one pass
  if (D == 64 && G == 1 && 5 * p.BH >= 4 * sms) return launch_fused(p);

  cudaError_t e = build_smem<D>();
  if (e != cudaSuccess) return e;
  e = ensure_smem_optin((const void *)global_read_tc<D>, (int)ReadLayout<D>::Bytes);
  if (e != cudaSuccess) return e;

  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)G;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3((unsigned)G, (unsigned)p.BH);
  cfg.blockDim = dim3(kBuildThreads);
  cfg.dynamicSmemBytes = BuildLayout<D>::Bytes;
  cfg.stream = p.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  {
    LaunchTimer timer(kKGlobalState, p.stream);
    e = cudaLaunchKernelEx(&cfg, global_build_tc<D>, bp);
    if (e == cudaSuccess) e = cudaGetLastError();
    timer.done(e);
  }
  if (e != cudaSuccess) return e;
  count_launch();

  rp.S = p.S;
  rp.z = p.z;
  rp.N = p.N;
  rp.tiles_per_head = (int)((p.N + 127) / 128);
  rp.total_tiles = (long)rp.tiles_per_head * p.BH;
  rp.eps = p.eps;
  const unsigned grid = (unsigned)std::min<long>(rp.total_tiles, sms);
  {
    // starts early beside the build (programmatic dependent launch): Q loads and
    // phi(Q) overlap the build's tail; S and z are read only after it completes
    LaunchTimer timer(kKGlobalRead, p.stream);
    cudaLaunchConfig_t rc = {};
    cudaLaunchAttribute ra[1];
    ra[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    ra[0].val.programmaticStreamSerializationAllowed = 1;
    rc.gridDim = dim3(grid);
    rc.blockDim = dim3(kReadThreads);
    rc.dynamicSmemBytes = ReadLayout<D>::Bytes;
    rc.stream = p.stream;
    rc.attrs = ra;
    rc.numAttrs = 1;
    e = cudaLaunchKernelEx(&rc, global_read_tc<D>, rp);
    if (e == cudaSuccess) e = cudaGetLastError();
    timer.done(e);
  }
  if (e == cudaSuccess) count_launch();
  return e;
}

}  // namespace

bool global_tc_supported(const Problem &p) {
  const DeviceInfo &di = device_info(-1);
  return p.dt == LA_BF16 && p.dk == p.dv && (p.dk == 64 || p.dk == 128) && p.N >= 1 && p.N <= 0x7fffffffL &&
         p.BH <= 65535 && di.cc_major == 10 && di.cc_minor == 3 && tensor_map_encoder() != nullptr;
}

cudaError_t launch_global_tc(const Problem &p) { return p.dk == 64 ? launch_t<64>(p) : launch_t<128>(p); }

cudaError_t launch_range_states(const Problem &p, long range_tokens, int ranges_per_head, int ctas, int pieces_per_cta,
                                float *piece_S, float *piece_z, int kernel_id, const float *log2g, int ret_H,
                                int mode) {
  if (p.dt != LA_BF16 || p.dk != 128 || p.dv != 128 || range_tokens % 64 != 0 || ranges_per_head < 1 || ctas < 1 ||
      pieces_per_cta < 1 || pieces_per_cta > 2 || (log2g && (ret_H < 1 || ret_H > kMaxRetentionHeads)))
    return cudaErrorInvalidValue;
  const long range_units = range_tokens / 64;
  const long units_total = (long)p.BH * ranges_per_head * range_units;
  // a CTA's run may span at most one range boundary; one piece a CTA needs runs that divide the ranges
  if ((units_total + ctas - 1) / ctas > range_units || ctas > units_total) return cudaErrorInvalidValue;
  if (pieces_per_cta == 1 && (units_total % ctas != 0 || range_units % (units_total / ctas) != 0))
    return cudaErrorInvalidValue;
  BuildParams bp;
  if (!make_map(&bp.tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.k, p.BH, p.N, 128, 64, 64) ||
      !make_map(&bp.tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.v, p.BH, p.N, 128, 64, 64))
    return cudaErrorInvalidValue;
  bp.S = bp.z = nullptr;
  bp.part_S = piece_S;
  bp.part_z = piece_z;
  bp.N = p.N;
  bp.units = (int)((p.N + 63) / 64);
  bp.units_total = units_total;
  bp.range_units = (int)range_units;
  bp.ranges_per_head = ranges_per_head;
  bp.pieces_per_cta = pieces_per_cta;
  bp.ret_H = log2g ? ret_H : 0;
  for (int h = 0; h < kMaxRetentionHeads; ++h) bp.log2g[h] = log2g && h < ret_H ? log2g[h] : 0.f;
  if ((mode == kModeRetention) != (log2g != nullptr)) return cudaErrorInvalidValue;
  cudaError_t e = mode == kModeRetention  ? build_smem<128, kModeRetention>()
                  : mode == kModeIdentity ? build_smem<128, kModeIdentity>()
                                          : build_smem<128>();
  if (e != cudaSuccess) return e;
  LaunchTimer timer(kernel_id, p.stream);
  if (mode == kModeRetention)
    global_build_tc<128, kModeRetention>
        <<<(unsigned)ctas, kBuildThreads, BuildLayout<128, true>::Bytes, p.stream>>>(bp);
  else if (mode == kModeIdentity)
    global_build_tc<128, kModeIdentity><<<(unsigned)ctas, kBuildThreads, BuildLayout<128>::Bytes, p.stream>>>(bp);
  else
    global_build_tc<128><<<(unsigned)ctas, kBuildThreads, BuildLayout<128>::Bytes, p.stream>>>(bp);
  e = cudaGetLastError();
  timer.done(e);
  if (e == cudaSuccess) count_launch();
  return e;
}

cudaError_t read_and_clear_global_tc_status(unsigned int *value) {
  const unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(value, g_global_status, sizeof(unsigned int));
  if (e == cudaSuccess && *value) e = cudaMemcpyToSymbol(g_global_status, &zero, sizeof(unsigned int));
  return e;
}

}  // namespace la
