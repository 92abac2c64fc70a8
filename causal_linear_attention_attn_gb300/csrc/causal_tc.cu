// Chunked causal linear attention on the sm_103a tensor cores (tcgen05, TMEM, TMA).
//
// The causal recurrence S_t = S_{t-1} + phi(k_t) v_t^T, z_t = z_{t-1} + phi(k_t),
// o_t = phi(q_t)^T S_t / (phi(q_t)^T z_t + eps) ("线性注意力从头到尾讲清楚" §7;
// "Linear Attention Math", "The recurrent form") is evaluated over chunks of
// C = 128 tokens: a chunk reads the state carried in from earlier chunks and
// adds its own masked pairwise part, then folds its keys and values into the
// state ("Linear Attention: From Pairwise Reads to a Recurrent State", "A
// recurrence need not force token-serial training").  Per chunk, with
// Q = phi(q), K = phi(k) rounded to bf16:
//   P      = tril(Q K^T)                    128x128x128 MMA, fp32 in TMEM
//   P_hi   = bf16(P), P_lo = bf16(P - P_hi) (the weights carry ~16 bits)
//   num    = Q bf16(S_prev) + P_hi V + P_lo V      3 MMAs into one TMEM tile
//   den    = Q . z_prev (fp32) + rowsum(P_hi + P_lo) + eps
//   S     += K^T V                          fp32 accumulator resident in TMEM
//   z     += column sums of K               fp32, CUDA cores
// d_k = d_v = 128.  The numerator and denominator use the same rounded
// weights, z never passes through bf16, and the state stays fp32.
//
// One CTA owns a contiguous segment of one head's tokens.  Long sequences are
// split into segments; a first pass (the range-state kernel of the global
// form) reduces K^T V and the key sums over parts of the earlier segments, and
// each segment starts from the sum of the parts before it.
//
// Warp roles (18 warps): 0 TMA producer; 1 MMA issuer and TMEM owner;
// 2-5 phi(Q) into tensor memory and the cross-chunk denominator phi(Q).z;
// 6-9 phi(K) in place and the column sums that advance z; 10-13 P split,
// denominator and bf16 state copy (and the final state); 14-17 normalised
// fp32 outputs through shared memory and TMA stores.  Every mbarrier wait is
// bounded; a wait that runs out raises the CTA abort word and the device
// status word, the CTA drains its in-flight copies and MMAs, frees TMEM and
// exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "per_device.h"
#include "tc_ptx.cuh"

namespace la {

__device__ unsigned int g_device_status;

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    else
      cudaGetLastError();
  });
  return fn;
}


namespace {
using namespace tc;

constexpr int kC = 128;               // tokens per chunk = MMA M
constexpr int kD = 128;               // d_k = d_v
constexpr uint32_t kBlk = 16384;      // one [128 rows x 64] bf16 block, 128-byte swizzled
constexpr uint32_t kTile = 2 * kBlk;  // [128 x 128] bf16 tile
constexpr int kThreads = 576;
constexpr int kWarpTma = 0, kWarpMma = 1, kWarpPhi = 2, kWarpEpi = 10, kWarpOut = 14;
constexpr uint32_t kBarOut = 4;  // named barrier of the output warps
constexpr int kPhiThreads = 256;  // feature-map warps 2-9
constexpr uint32_t kBarPhi = 1, kBarEpi = 2;  // named barrier ids
constexpr int kExact = 64;  // leading tokens of each head computed by the exact fp32 pass

struct Layout {
  static constexpr int kStages = 2;
  static constexpr uint32_t Q = 0;
  static constexpr uint32_t K = kStages * kTile;
  static constexpr uint32_t V = K + kStages * kTile;
  static constexpr uint32_t Sb = V + kStages * kTile;  // bf16 copy of the carried state
  static constexpr uint32_t DenX = Sb + kTile;          // phi(q).z per row, per stage
  static constexpr uint32_t Den = DenX + kStages * kC * 4;  // final denominators, 2 chunks
  static constexpr uint32_t Z = Den + 2 * kC * 4;
  static constexpr uint32_t Bars = Z + kD * 4;
  static constexpr int kNumBars = 34;
  static constexpr uint32_t Misc = Bars + kNumBars * 8;
  static constexpr uint32_t Bytes = Misc + 16;
  // The dynamic shared memory base follows the 1 KB reserved per block and is
  // 1024-aligned; the kernel checks this and refuses to run otherwise.
  static constexpr uint32_t Alloc = Bytes;
  static constexpr uint32_t TmemCols = 512;
};
static_assert(Layout::Alloc <= 232448, "shared memory budget");

// TMEM columns (main mode): S accumulator, P (fp32, then split bf16 hi/lo in
// place), the output accumulator, and two buffers of phi(Q) packed as bf16
// pairs (the A operand of Q K^T and Q S).
constexpr uint32_t kColS = 0, kColP = 128, kColO = 256, kColQ = 384;
constexpr uint32_t kAbortMisaligned = 2u;  // status bit: shared memory base not 1024-aligned


struct TcParams {
  CUtensorMap tq, tk, tv;  // 3-D maps over [BH][N][128] bf16, box 64 x 128 x 1, 128-byte swizzle
  CUtensorMap to;          // 3-D map over the fp32 output [BH][N][128], box 32 x 128 x 1, 128-byte swizzle
  CUtensorMap to_tail;     // the same tensor, box 32 x 64 x 1: rows 64..127 of a head's first chunk
  float *out, *S_out, *z_out;
  const float *S0, *z0;      // initial state (nullable = zero)
  float *part_S, *part_z;    // first-pass pieces: [2 fp_ctas][128][128], [2 fp_ctas][128]
  long N;
  int seg_len, nseg;
  // first pass (see prefix_pieces): fp_ranges leading segments of every head,
  // fp_range_units 64-token units each, fp_units in all, cut into fp_ctas runs
  long fp_units;
  int fp_ctas, fp_range_units, fp_ranges, fp_pieces_per_cta;
  int n_exact;
  float eps;
  // retention (decayed state, no denominator): log2 of the decay of head h % ret_H
  int ret_H;
  float log2g[kMaxRetentionHeads];
  // how long an mbarrier wait may take before the CTA gives up (kWaitNs unless a
  // test armed la_test_inject_missing_load), and the chunk whose key load CTA
  // (0, 0) leaves out on such a test launch (-1: none)
  unsigned long long wait_ns;
  int skip_k_chunk;
};

__device__ __forceinline__ float dot8(uint4 y, const float *z) {
  const uint32_t w[4] = {y.x, y.y, y.z, y.w};
  const float4 z0 = *reinterpret_cast<const float4 *>(z), z1 = *reinterpret_cast<const float4 *>(z + 4);
  const float2 zz[4] = {make_float2(z0.x, z0.y), make_float2(z0.z, z0.w), make_float2(z1.x, z1.y),
                        make_float2(z1.z, z1.w)};
  float2 s = make_float2(0.f, 0.f);  // even and odd features, one packed FMA per pair
#pragma unroll
  for (int e = 0; e < 4; ++e)
    s = __ffma2_rn(make_float2(__uint_as_float(w[e] << 16), __uint_as_float(w[e] & 0xffff0000u)), zz[e], s);
  return s.x + s.y;
}

// Write 32 values (columns col0 .. col0+31 of row `row`) as bf16 into a
// [128 x 128] tile made of two 64-column swizzled blocks.
__device__ __forceinline__ void store_row32_bf16(uint8_t *tile, int row, int col0, const uint32_t (&r)[32]) {
  uint8_t *blk = tile + (col0 >> 6) * kBlk;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int c = (col0 & 63) + q * 8;
    const float *v = reinterpret_cast<const float *>(r) + 8 * q;
    *reinterpret_cast<uint4 *>(blk + sw128_offset(row, c)) =
        make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]), pack_bf16(v[6], v[7]));
  }
}

// As store_row32_bf16, as a bf16 pair: hi = bf16(x) into `hi`, lo = bf16(x - hi) into `lo`.
__device__ __forceinline__ void store_row32_split(uint8_t *hi, uint8_t *lo, int row, int col0,
                                                  const uint32_t (&r)[32]) {
  const int off = (col0 >> 6) * kBlk;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int c = (col0 & 63) + q * 8;
    const float *v = reinterpret_cast<const float *>(r) + 8 * q;
    uint32_t h[4], l[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      h[e] = pack_bf16(v[2 * e], v[2 * e + 1]);
      l[e] = pack_bf16(v[2 * e] - __uint_as_float(h[e] << 16), v[2 * e + 1] - __uint_as_float(h[e] & 0xffff0000u));
    }
    *reinterpret_cast<uint4 *>(hi + off + sw128_offset(row, c)) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4 *>(lo + off + sw128_offset(row, c)) = make_uint4(l[0], l[1], l[2], l[3]);
  }
}

// Four fp32 values (as raw bits) times f, by two packed multiplies.
__device__ __forceinline__ float4 scale4(const uint32_t *r, float f) {
  const float2 a = __fmul2_rn(make_float2(__uint_as_float(r[0]), __uint_as_float(r[1])), make_float2(f, f));
  const float2 b = __fmul2_rn(make_float2(__uint_as_float(r[2]), __uint_as_float(r[3])), make_float2(f, f));
  return make_float4(a.x, a.y, b.x, b.y);
}

// K-major operand (rows of 64 K-elements): k-step ks covers K elements [16ks, 16ks+16).
__device__ __forceinline__ uint64_t kdesc(uint32_t tile, int ks) {
  return sw128_desc(tile + (ks >> 2) * kBlk + (ks & 3) * 32, 16, 1024);
}
// MN-major operand (rows = K index, 64 M/N elements per row, two 64-wide blocks).
__device__ __forceinline__ uint64_t mndesc(uint32_t tile, int ks) {
  return sw128_desc(tile + ks * 2048, kBlk, 1024);
}

// Column sums of the valid rows of a [128 x 128] bf16 tile over eight warps:
// warp `w` adds columns [16w, 16w+16); lane l takes the pair 16w + 2(l&7) over
// rows t = (l>>3) mod 4, and the four row phases meet through two shuffles.
// Lanes l < 8 return the sums of columns (c, c+1).
__device__ __forceinline__ int column_pair_sums_8w(const uint8_t *tile, int w, int lane, int rows, float &s0,
                                                   float &s1) {
  const int c = 16 * w + 2 * (lane & 7);
  const int ph = lane >> 3;
  const uint8_t *blk = tile + (c >> 6) * kBlk;
  const int cc = c & 63;
  const uint32_t off0 = sw128_offset(ph, cc), off1 = sw128_offset(ph + 4, cc);
  float2 a = make_float2(0.f, 0.f);  // the pair's two columns, packed adds
  const int full = rows >> 3;
#pragma unroll 4
  for (int g = 0; g < full; ++g) {
    const uint32_t x = *reinterpret_cast<const uint32_t *>(blk + g * 1024 + off0);
    const uint32_t y = *reinterpret_cast<const uint32_t *>(blk + g * 1024 + off1);
    a = __fadd2_rn(a, __fadd2_rn(make_float2(__uint_as_float(x << 16), __uint_as_float(x & 0xffff0000u)),
                                 make_float2(__uint_as_float(y << 16), __uint_as_float(y & 0xffff0000u))));
  }
  float a0 = a.x, a1 = a.y;
  for (int t = 8 * full + ph; t < rows; t += 4) {
    const uint32_t x = *reinterpret_cast<const uint32_t *>(blk + sw128_offset(t, cc));
    a0 += __uint_as_float(x << 16);
    a1 += __uint_as_float(x & 0xffff0000u);
  }
  a0 += __shfl_xor_sync(0xffffffffu, a0, 8);
  a1 += __shfl_xor_sync(0xffffffffu, a1, 8);
  a0 += __shfl_xor_sync(0xffffffffu, a0, 16);
  a1 += __shfl_xor_sync(0xffffffffu, a1, 16);
  s0 = a0;
  s1 = a1;
  return c;
}

// The first pass cut the leading segments of all heads, one after another,
// into fp_ctas even runs of units, each at most one segment long.  With two
// pieces a run, run c's part in its first segment is piece 2c and the rest
// piece 2c + 1 (all zeros when the run stays in one segment); with one piece a
// run, the runs divide the segments and run c is piece c.  Pieces are in unit
// order, and head bh's segments [0, seg) are exactly the pieces [first, last]
// returned here.
struct PieceRange {
  long first, last;
};
__device__ __forceinline__ PieceRange prefix_pieces(const TcParams &p, int bh, int seg) {
  const long L = p.fp_range_units, U = p.fp_units, C = p.fp_ctas;
  const long ub = (long)bh * p.fp_ranges * L, ue = ub + (long)seg * L;  // units [ub, ue)
  if (p.fp_pieces_per_cta == 1) {
    const long run = U / C;
    return PieceRange{ub / run, ue / run - 1};
  }
  // the runs holding units ub and ue - 1
  long c0 = max(0L, ub * C / U - 1);
  while (U * (c0 + 1) / C <= ub) ++c0;
  long c1 = max(c0, (ue - 1) * C / U - 1);
  while (U * (c1 + 1) / C <= ue - 1) ++c1;
  PieceRange r;
  r.first = 2 * c0 + (U * c0 / C < ub ? 1 : 0);  // run c0 crosses into segment rb at ub
  const long s1 = U * c1 / C;
  r.last = 2 * c1 + ((s1 / L + 1) * L <= ue - 1 ? 1 : 0);  // unit ue - 1 after run c1's crossing
  return r;
}

// Head-local end (in 64-token units) of first-pass piece `piece` of head bh.
__device__ __forceinline__ long piece_end_units(const TcParams &p, int bh, long piece) {
  const long L = p.fp_range_units, U = p.fp_units, C = p.fp_ctas;
  long e;
  if (p.fp_pieces_per_cta == 1) {
    e = (piece + 1) * (U / C);
  } else {
    const long c = piece >> 1, s0 = U * c / C, e0 = U * (c + 1) / C;
    e = (piece & 1) ? e0 : min(e0, (s0 / L + 1) * L);
  }
  return e - (long)bh * p.fp_ranges * L;
}

// kRet: retention instead of normalized linear attention.  With the decay
// gamma, a chunk of C valid tokens, chunk-local rows i (query) and j (key),
// key weights w_j = gamma^(C-1-j) and S the state before the chunk, tensor
// memory holds A = gamma^C S and
//   out_i = gamma^(i+1-C) (q_i A + sum_{j <= i} ((q_i . k_j) w_j) v_j)
//   S_new = A + (w k)^T V   (then times the next chunk's gamma^C)
// q and k are used as given, so the dot products cancel and every operand
// that is not an input goes to the tensor cores as a bf16 hi/lo pair:
// (q_i . k_j) w_j is split as P is; the weighted keys are split into the
// consumed Q slot (lo, as soon as Q is in tensor memory) and the K tile (hi,
// once Q K^T has read the raw keys).  The update takes the low parts first and
// the slot is reloaded as soon as they have been read (so Q has one stage);
// the copy of A that Q reads is split into Sb (hi) and the other Q slot (lo).  Every factor lies within 2^+-54 for gamma >= 0.75.  There is
// no z, no denominator and no exact leading-token pass.
// kModeIdentity: q and k are already features; they reach the MMAs as given,
// with the normalizer, denominators and no exact leading-token pass.  Given
// features can be heavy-tailed (a few keys dominate each read while the state
// sums all of them), so this mode too reads the carried state as a hi/lo pair.
template <int kMode>
__global__ void __maxnreg__(96) causal_tc_kernel(const __grid_constant__ TcParams p) {
  constexpr bool kRet = kMode == kModeRetention, kRaw = kMode != kModeElu;
  // one Q slot; the other holds the low parts of the state copy read by the queries
  constexpr bool kQ1 = kMode != kModeElu, kSplitS = kQ1;
  using Lay = Layout;
  constexpr int kStages = Lay::kStages;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {  // the swizzled tiles need a 1024-byte aligned base
    if (threadIdx.x == 0) atomicOr(&g_device_status, kAbortMisaligned);
    return;
  }
  uint8_t *sm = smem_raw;
  float *den_x = reinterpret_cast<float *>(sm + Lay::DenX);
  float *den_s = reinterpret_cast<float *>(sm + Lay::Den);
  float *zs = reinterpret_cast<float *>(sm + Lay::Z);
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + Lay::Bars);
  // per stage: Q landed, K landed, V landed, phi applied, raw Q consumed, K free, V free
  uint64_t *full_q = bars, *full_k = bars + 3, *full_v = bars + 6, *phi_done = bars + 9, *q_empty = bars + 12,
           *k_empty = bars + 15, *v_empty = bars + 18;
  uint64_t *s_full = bars + 21, *pp_ready = bars + 22, *o_full = bars + 23, *sb_ready = bars + 24,
           *o_free = bars + 25, *drain = bars + 26, *p_full = bars + 27, *den_ready = bars + 28,  // [2]
           *qt_free = bars + 30,  // [2]: phi(Q) tensor-memory buffers
           *k_ready = bars + 32,  // retention: high parts of the weighted keys in place
           *klo_ready = bars + 33;  // retention: their low parts in the Q slot
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + Lay::Misc);
  volatile uint32_t *abort_word = reinterpret_cast<volatile uint32_t *>(sm + Lay::Misc + 4);
  unsigned int *status = &g_device_status;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.y;
  const long t_begin = (long)blockIdx.x * p.seg_len;
  const long t_end = min(p.N, t_begin + p.seg_len);
  const int seg = blockIdx.x;  // segments before this one arrive as first-pass pieces
  const bool last_seg = (int)blockIdx.x == p.nseg - 1;
  const int nchunks = (int)((t_end - t_begin + kC - 1) / kC);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_q[s], 1);
      mbar_init(&full_k[s], 1);
      mbar_init(&full_v[s], 1);
      mbar_init(&phi_done[s], kPhiThreads);
      mbar_init(&q_empty[s], kRet ? 1 : kPhiThreads);  // retention: the state update's commit
      // the MMA commit plus the epilogue's 128 threads once they have read den_x[s]
      mbar_init(&k_empty[s], 129);
      mbar_init(&v_empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(pp_ready, 128);
    mbar_init(o_full, 1);
    mbar_init(sb_ready, 128);
    mbar_init(o_free, 128);
    mbar_init(drain, 1);
    mbar_init(&qt_free[0], 1);
    mbar_init(&qt_free[1], 1);
    mbar_init(p_full, 1);
    mbar_init(&den_ready[0], 128);
    mbar_init(&den_ready[1], 128);
    mbar_init(k_ready, kPhiThreads);
    mbar_init(klo_ready, kPhiThreads);
    *abort_word = 0;
    fence_barrier_init();
  }
  if (warp == kWarpMma) tmem_alloc(tmem_slot, Lay::TmemCols);
  // the exact leading-token pass queued after this kernel may start on the SMs this grid leaves free
  if (threadIdx.x == 0) pdl_trigger();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kWarpTma) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      prefetch_tmap(&p.tq);
      prefetch_tmap(&p.tk);
      prefetch_tmap(&p.tv);
      int issued_q = 0, issued_k = 0, issued_v = 0;
      // a test launch (la_test_inject_missing_load) leaves out one key load of CTA (0, 0): the
      // consumers' bounded waits then run out, and the CTA drains and exits with the timeout set
      const int skip_k = blockIdx.x == 0 && blockIdx.y == 0 ? p.skip_k_chunk : -1;
      // Q of chunk c: stage c % 2, or (retention) always slot 0, once the previous chunk's state
      // update has read the low parts of its weighted keys there
      auto load_q = [&](int c, int tok) -> bool {
        const int qs = kQ1 ? 0 : c % kStages;
        if (kQ1 ? c >= 1 : c >= kStages) {
          const uint32_t ph = kQ1 ? (uint32_t)(c - 1) & 1 : (uint32_t)(c / kStages - 1) & 1;
          if (!mbar_wait(&q_empty[qs], ph, abort_word, status, p.wait_ns)) return false;
        }
        mbar_arrive_expect_tx(&full_q[qs], kTile);
        tma_load_3d(sm + Lay::Q + qs * kTile, &p.tq, &full_q[qs], 0, tok, bh);
        tma_load_3d(sm + Lay::Q + qs * kTile + kBlk, &p.tq, &full_q[qs], 64, tok, bh);
        issued_q = c + 1;
        return true;
      };
      for (int c = 0; c < nchunks; ++c) {
        const int s = c % kStages;
        const uint32_t u = c / kStages;
        const int tok = (int)(t_begin + (long)c * kC);
        if (!kRet && !load_q(c, tok)) break;
        if (c >= kStages && !mbar_wait(&k_empty[s], (u - 1) & 1, abort_word, status, p.wait_ns)) break;
        if (c != skip_k) {
          mbar_arrive_expect_tx(&full_k[s], kTile);
          tma_load_3d(sm + Lay::K + s * kTile, &p.tk, &full_k[s], 0, tok, bh);
          tma_load_3d(sm + Lay::K + s * kTile + kBlk, &p.tk, &full_k[s], 64, tok, bh);
        }
        issued_k = c + 1;
        // retention: Q's single slot frees before this V stage does (the stage is also the output
        // staging of the chunk two back), so Q goes first
        if (kRet && !load_q(c, tok)) break;
        if (c >= kStages && !mbar_wait(&v_empty[s], (u - 1) & 1, abort_word, status, p.wait_ns)) break;
        mbar_arrive_expect_tx(&full_v[s], kTile);
        tma_load_3d(sm + Lay::V + s * kTile, &p.tv, &full_v[s], 0, tok, bh);
        tma_load_3d(sm + Lay::V + s * kTile + kBlk, &p.tv, &full_v[s], 64, tok, bh);
        issued_v = c + 1;
      }
      // every issued copy must land before shared memory is released
      for (int c = max(0, issued_q - (kQ1 ? 1 : kStages)); c < issued_q; ++c)
        wait_drain(&full_q[kQ1 ? 0 : c % kStages], kQ1 ? (uint32_t)c & 1 : (uint32_t)(c / kStages) & 1, status);
      for (int c = max(0, issued_k - kStages); c < issued_k; ++c)
        if (c != skip_k) wait_drain(&full_k[c % kStages], (c / kStages) & 1, status);
      for (int c = max(0, issued_v - kStages); c < issued_v; ++c)
        wait_drain(&full_v[c % kStages], (c / kStages) & 1, status);
    }
  } else if (warp == kWarpMma) {
    // ---------------- MMA issuer (one thread) ----------------
    // This warp shares its scheduler with busy feature-map and epilogue warps, so the loop
    // overhead between MMAs sets the issue rate: the loops are unrolled by 4 (measured faster
    // than by 1, 2 or 8 at 4 x 16 x 8192).
    if (lane == 0) {
      const uint32_t tO = tmem + kColO, tS = tmem + kColS, tP = tmem + kColP;
      constexpr uint32_t iKK = idesc_bf16_f32(128, 128, 0, 0);
      constexpr uint32_t iKM = idesc_bf16_f32(128, 128, 0, 1);
      constexpr uint32_t iMM = idesc_bf16_f32(128, 128, 1, 1);
      const uint32_t sK = smem_u32(sm + Lay::K), sV = smem_u32(sm + Lay::V), sSb = smem_u32(sm + Lay::Sb);
      // retention: low parts of the weighted keys (Q slot 0) and of the state copy (Q slot 1)
      const uint32_t sKlo = smem_u32(sm + Lay::Q), sSblo = smem_u32(sm + Lay::Q + kTile);
      for (int c = 0; c < nchunks; ++c) {
        const int s = c % kStages;
        const uint32_t u = c / kStages;
        if (!mbar_wait(&phi_done[s], u & 1, abort_word, status, p.wait_ns)) break;
        // retention: the keys reach Q K^T as loaded (no in-place pass before it)
        if (kRet && !mbar_wait(&full_k[s], u & 1, abort_word, status, p.wait_ns)) break;
        const uint32_t k = sK + s * kTile, v = sV + s * kTile;
        const uint32_t tQ = tmem + kColQ + 64 * (c & 1);
        // The single P tile is free for this chunk's Q K^T: the P-split warps finished with the
        // previous chunk's P before its P V was issued, and this thread's MMAs execute in issue
        // order, so that P V reads P before Q K^T writes it (no wait, no drain of the pipe).
        tc_fence_after();
        // P = Q K^T, phi(Q) from tensor memory (8 columns per 16 features)
#pragma unroll 4
        for (int ks = 0; ks < 8; ++ks) mma_bf16_ts(tP, tQ + 8 * ks, kdesc(k, ks), iKK, ks > 0);
        mma_commit(p_full);
        // V is first read by the state update (Q K^T does not need it)
        if (!mbar_wait(&full_v[s], u & 1, abort_word, status, p.wait_ns)) break;
        // S += K^T V; retention: the weighted keys as a pair, the low parts (in the Q slot) first
        // so that the slot is released for the next chunk's Q as early as possible
        auto state_update = [&](uint32_t a) {
#pragma unroll 4
          for (int ks = 0; ks < 8; ++ks) mma_bf16(tS, mndesc(a, ks), mndesc(v, ks), iMM, 1);
        };
        // O = Q bf16(S_prev) (pair modes: hi and lo of the state copy)
        auto state_read = [&]() {
#pragma unroll 4
          for (int ks = 0; ks < 8; ++ks) mma_bf16_ts(tO, tQ + 8 * ks, mndesc(sSb, ks), iKM, ks > 0);
          if (kSplitS) {
#pragma unroll 4
            for (int ks = 0; ks < 8; ++ks) mma_bf16_ts(tO, tQ + 8 * ks, mndesc(sSblo, ks), iKM, 1);
          }
          mma_commit(&qt_free[c & 1]);
        };
        // The read needs the copy of the previous state and the previous outputs read out; the
        // update needs that copy taken and (retention) the keys weighted.  Retention runs the
        // read between the two halves of the update, while the keys' high parts are formed.
        if (!mbar_wait(sb_ready, c & 1, abort_word, status, p.wait_ns)) break;
        if (kRet) {
          if (!mbar_wait(klo_ready, c & 1, abort_word, status, p.wait_ns)) break;
          tc_fence_after();
          state_update(sKlo);
          mma_commit(&q_empty[0]);  // the Q slot may take the next chunk's Q
          if (c > 0 && !mbar_wait(o_free, (c - 1) & 1, abort_word, status, p.wait_ns)) break;
          tc_fence_after();
          state_read();
          if (!mbar_wait(k_ready, c & 1, abort_word, status, p.wait_ns)) break;
          tc_fence_after();
          state_update(k);
        } else {
          tc_fence_after();
          state_update(k);
          if (c > 0 && !mbar_wait(o_free, (c - 1) & 1, abort_word, status, p.wait_ns)) break;
          tc_fence_after();
          state_read();
        }
        mma_commit(s_full);  // the update is complete and the copy has been read
        mma_commit(&k_empty[s]);
        if (!mbar_wait(pp_ready, c & 1, abort_word, status, p.wait_ns)) break;
        tc_fence_after();
        // O += P_hi V + P_lo V, P read from tensor memory: for keys [16ks, 16ks+16)
        // columns 16ks..16ks+7 hold P_hi and 16ks+8..16ks+15 hold P_lo
#pragma unroll 4
        for (int ks = 0; ks < 8; ++ks) {
          mma_bf16_ts(tO, tP + 16 * ks, mndesc(v, ks), iKM, 1);
          mma_bf16_ts(tO, tP + 16 * ks + 8, mndesc(v, ks), iKM, 1);
        }
        mma_commit(o_full);
      }
      mma_commit(drain);
      wait_drain(drain, 0, status);
    }
  } else if (warp < kWarpEpi) {
    // ---------------- feature-map warps (8) ----------------
    // Warp w takes rows 32*(w%4) .. +31 (its tensor-memory lane quarter) and
    // the 64-feature half (w-2)/4 of both the Q and the K tile.
    const int pt = threadIdx.x - kWarpPhi * 32;  // 0..255
    const int quarter = warp & 3;
    const int half = (warp - kWarpPhi) >> 2;
    const int row = quarter * 32 + lane;
    const float lg = kRet ? p.log2g[bh % max(p.ret_H, 1)] : 0.f;  // retention: log2 gamma
    if (seg > 0 && !kRet) pdl_wait();  // the first pass's pieces are complete and visible
    if (!kRet && pt < kD) {
      // first-pass pieces start from zero; a segment starts from the caller's state plus them
      float z = p.z0 ? p.z0[(long)bh * kD + pt] : 0.f;
      if (seg > 0) {
        const PieceRange pr = prefix_pieces(p, bh, seg);
        for (long piece = pr.first; piece <= pr.last; ++piece) z += p.part_z[piece * kD + pt];
      }
      zs[pt] = z;
      den_x[pt] = den_x[kC + pt] = 0.f;
    }
    if (kRet && pt < kD) den_x[pt] = den_x[kC + pt] = 0.f;
    named_bar(kBarPhi, kPhiThreads);
    for (int c = 0; c < nchunks; ++c) {
      const int s = c % kStages;
      const uint32_t u = c / kStages;
      const int tv = (int)min((long)kC, t_end - (t_begin + (long)c * kC));
      uint8_t *Kt = sm + Lay::K + s * kTile;
      bool ok = mbar_wait(&full_k[s], u & 1, abort_word, status, p.wait_ns);
      ok = ok && mbar_wait(&full_q[kQ1 ? 0 : s], kQ1 ? (uint32_t)c & 1 : u & 1, abort_word, status, p.wait_ns);
      // this chunk's phi(Q) buffer is free once Q K^T and Q S of the chunk two back have completed
      if (ok && c >= 2) ok = mbar_wait(&qt_free[c & 1], ((c >> 1) - 1) & 1, abort_word, status, p.wait_ns);
      if (bar_or(kBarPhi, kPhiThreads, !ok)) break;
      {
        // phi(Q) half row -> packed bf16 pairs -> tensor memory; the partial phi(q).z_prev
        // from the same rounded values meets its other half in shared memory
        const uint8_t *Qb = sm + Lay::Q + (kQ1 ? 0 : s) * kTile + half * kBlk;
        const uint32_t tq = tmem + ((uint32_t)(quarter * 32) << 16) + kColQ + 64 * (c & 1) + 32 * half;
        float dx = 0.f;
#pragma unroll 1
        for (int g = 0; g < 2; ++g) {
          uint4 xv[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) xv[e] = *reinterpret_cast<const uint4 *>(Qb + sw128_offset(row, g * 32 + e * 8));
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint4 y = kRaw ? xv[e] : phi8(xv[e]);
            w[4 * e] = y.x, w[4 * e + 1] = y.y, w[4 * e + 2] = y.z, w[4 * e + 3] = y.w;
            if (!kRet) dx += dot8(y, zs + half * 64 + g * 32 + e * 8);
          }
          tmem_st16(tq + 16 * g, w);
        }
        if (!kRet) {
          atomicAdd(&den_x[s * kC + row], dx);
          mbar_arrive(&q_empty[kQ1 ? 0 : s]);  // raw Q consumed
        }
      }
      // phi(K) half row in place (all loads of a step first: the in-place stores would order them);
      // retention: the raw keys times their state weight w_row as a bf16 pair, the low parts into
      // the consumed Q slot (part 1) and, once Q K^T has read the raw keys, the high parts in
      // place (part 2)
      auto transform_k = [&](float wk, int part) {
        uint8_t *Kb = Kt + half * kBlk, *Lb = sm + Lay::Q + half * kBlk;
#pragma unroll 1
        for (int g = 0; g < 2; ++g) {
          uint4 kv[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) kv[e] = *reinterpret_cast<const uint4 *>(Kb + sw128_offset(row, g * 32 + e * 8));
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint32_t off = sw128_offset(row, g * 32 + e * 8);
            if (kRet) {
              uint4 hi, lo;
              split8(kv[e], wk, hi, lo);
              if (part == 1)
                *reinterpret_cast<uint4 *>(Lb + off) = lo;
              else
                *reinterpret_cast<uint4 *>(Kb + off) = hi;
            } else {
              *reinterpret_cast<uint4 *>(Kb + off) = phi8(kv[e]);
            }
          }
        }
      };
      if (!kRaw) transform_k(1.f, 0);
      named_bar(kBarPhi, kPhiThreads);  // every K row transformed; every read of zs done
      if (!kRet) {
        // column sums of phi(K) over the valid rows (bf16 values, as the MMA sees them)
        float s0, s1;
        const int col = column_pair_sums_8w(Kt, warp - kWarpPhi, lane, tv, s0, s1);
        if (lane < 8) {
          zs[col] += s0;
          zs[col + 1] += s1;
        }
      }
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&phi_done[s]);
      if (kRet) {
        // every raw Q read of this slot is done (the barrier above): the low parts may go in
        const float wk = exp2f((float)(tv - 1 - row) * lg);
        transform_k(wk, 1);
        fence_async_smem();
        mbar_arrive(klo_ready);
        const bool okp = mbar_wait(p_full, c & 1, abort_word, status, p.wait_ns);  // Q K^T has read the raw keys
        if (bar_or(kBarPhi, kPhiThreads, !okp)) break;
        transform_k(wk, 2);
        fence_async_smem();
        mbar_arrive(k_ready);
      }
      named_bar(kBarPhi, kPhiThreads);  // z complete before the next chunk reads it
    }
    if (!kRet && !*abort_word && pt < kD) {
      if (last_seg) p.z_out[(long)bh * kD + pt] = zs[pt];
    }
  } else if (warp < kWarpOut) {
    // ---------------- P split, denominator and state copy (warps 10-13) ----------------
    const int quarter = warp & 3;
    const int T = quarter * 32 + lane;  // TMEM lane: chunk row (token) or state row (feature)
    const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
    uint32_t r[32];
    bool ok = true;
    {
      uint8_t *Sb = sm + Lay::Sb;
      if (seg > 0) pdl_wait();  // the first pass's pieces are complete and visible
      // initial state: caller's state plus the first-pass pieces before this segment
      // (retention: each decayed over the tokens from its end to the segment start)
      // (retention: tensor memory holds the state times gamma^C of the chunk about to be read)
      const PieceRange pr = seg > 0 ? prefix_pieces(p, bh, seg) : PieceRange{0, -1};
      const float lg = kRet ? p.log2g[bh % max(p.ret_H, 1)] : 0.f;
      const float c0 = (float)min((long)kC, t_end - t_begin);
      if (kRet) den_s[T] = exp2f((float)(kC - 1 - T) * lg);  // key weights gamma^(127-j), in the denominators' slot
      for (int cb = 0; cb < 4; ++cb) {
        float v[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = 0.f;
        if (p.S0) {
          const float4 *src = reinterpret_cast<const float4 *>(p.S0 + ((long)bh * kD + T) * kD + cb * 32);
          const float f = kRet ? exp2f(((float)t_begin + c0) * lg) : 1.f;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float4 x = src[e];
            v[4 * e] += f * x.x, v[4 * e + 1] += f * x.y, v[4 * e + 2] += f * x.z, v[4 * e + 3] += f * x.w;
          }
        }
        for (long piece = pr.first; piece <= pr.last; ++piece) {
          const float4 *src = reinterpret_cast<const float4 *>(p.part_S + (piece * kD + T) * kD + cb * 32);
          const float f = kRet ? exp2f(((float)(t_begin - 64 * piece_end_units(p, bh, piece)) + c0) * lg) : 1.f;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float4 x = src[e];
            v[4 * e] += f * x.x, v[4 * e + 1] += f * x.y, v[4 * e + 2] += f * x.z, v[4 * e + 3] += f * x.w;
          }
        }
#pragma unroll
        for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(v[e]);
        tmem_st32(tl + kColS + cb * 32, r);
        if (kSplitS)
          store_row32_split(Sb, sm + Lay::Q + kTile, T, cb * 32, r);
        else
          store_row32_bf16(Sb, T, cb * 32, r);
      }
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(sb_ready);

      for (int c = 0; c < nchunks; ++c) {
        const int s = c % kStages;
        const uint32_t u = c / kStages;
        const long tok = t_begin + (long)c * kC;
        const int tv = (int)min((long)kC, t_end - tok);
        const uint32_t tP = tl + kColP;
        bool w = mbar_wait(&phi_done[s], u & 1, abort_word, status, p.wait_ns) &&
                 mbar_wait(p_full, c & 1, abort_word, status, p.wait_ns);
        if (bar_or(kBarEpi, 128, !w)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // retention: key j's weight gamma^(tv-1-j) = table[j] * gamma^(tv-128)
        const float wc = kRet ? exp2f((float)(tv - kC) * lg) : 1.f;
        float den = den_x[s * kC + T];
        den_x[s * kC + T] = 0.f;  // the feature-map warps accumulate the next use of this slot
        mbar_arrive(&k_empty[s]);
        // P -> causal mask -> bf16 hi/lo, written back over the same columns:
        // keys [16g, 16g+16) become 8 columns of P_hi pairs then 8 of P_lo pairs.
        // Key blocks right of this warp's rows are all masked (zeros).
        float2 rs2 = make_float2(0.f, 0.f);  // row sum over even and odd keys
        const int jmax = min(T, tv - 1);       // key j is kept when j <= T (inclusive) and j < tv
#pragma unroll 1
        for (int cb = 0; cb < 4; ++cb) {
          if (cb > quarter) {
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = 0u;
          } else {
            tmem_ld32(tP + cb * 32, r);
#pragma unroll
            for (int g = 0; g < 2; ++g) {
              uint32_t o[16];
#pragma unroll
              for (int m = 0; m < 8; ++m) {
                const int j = cb * 32 + g * 16 + 2 * m;
                float p0 = j <= jmax ? __uint_as_float(r[g * 16 + 2 * m]) : 0.f;
                float p1 = j + 1 <= jmax ? __uint_as_float(r[g * 16 + 2 * m + 1]) : 0.f;
                float2 pp = make_float2(p0, p1);  // packed fp32 pairs from here on
                if (kRet) {
                  const float2 wj = *reinterpret_cast<const float2 *>(den_s + j);
                  pp = __fmul2_rn(pp, __fmul2_rn(wj, make_float2(wc, wc)));
                }
                const uint32_t hw = pack_bf16(pp.x, pp.y);
                const float2 hh = make_float2(__uint_as_float(hw << 16), __uint_as_float(hw & 0xffff0000u));
                const float2 ll = __ffma2_rn(hh, make_float2(-1.f, -1.f), pp);  // pp - hh, exact
                const uint32_t lw = pack_bf16(ll.x, ll.y);
                rs2 = __fadd2_rn(rs2, pp);  // the row sum equals that of hi + lo to within 2^-16 relative
                o[m] = hw;
                o[8 + m] = lw;
              }
#pragma unroll
              for (int e = 0; e < 16; ++e) r[g * 16 + e] = o[e];
            }
          }
          tmem_st32(tP + cb * 32, r);
        }
        den = (den + (rs2.x + rs2.y)) + p.eps;
        if (!kRet) den_s[(c & 1) * kC + T] = den;
        tc_fence_before();
        mbar_arrive(pp_ready);
        mbar_arrive(&den_ready[c & 1]);
        // bf16 copy of the updated state for the next chunk's cross read
        w = mbar_wait(s_full, c & 1, abort_word, status, p.wait_ns);
        if (bar_or(kBarEpi, 128, !w)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // retention: the state times the next chunk's gamma^C, in place, before the copy
        // (after the last chunk tensor memory keeps the final state itself)
        const float gC = kRet && c + 1 < nchunks ? exp2f((float)min((long)kC, t_end - tok - kC) * lg) : 1.f;
#pragma unroll 1
        for (int cb = 0; cb < 4; ++cb) {
          tmem_ld32(tl + kColS + cb * 32, r);
          if (kRet) {
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * gC);
            if (c + 1 < nchunks) tmem_st32(tl + kColS + cb * 32, r);
          }
          if (kSplitS)
            store_row32_split(Sb, sm + Lay::Q + kTile, T, cb * 32, r);
          else
            store_row32_bf16(Sb, T, cb * 32, r);
        }
        fence_async_smem();
        tc_fence_before();
        mbar_arrive(sb_ready);
      }
    }
    // final (or partial) state, fp32
    if (ok && !*abort_word && last_seg) {
      float *dst = p.S_out + ((long)bh * kD + T) * kD;
      for (int cb = 0; cb < 4; ++cb) {
        tmem_ld32(tl + kColS + cb * 32, r);
        float4 *d4 = reinterpret_cast<float4 *>(dst + cb * 32);
#pragma unroll
        for (int e = 0; e < 8; ++e)
          d4[e] = make_float4(__uint_as_float(r[4 * e]), __uint_as_float(r[4 * e + 1]),
                              __uint_as_float(r[4 * e + 2]), __uint_as_float(r[4 * e + 3]));
      }
    }
  } else {
    // ---------------- normalised outputs (warps 14-17) ----------------
    const int quarter = warp & 3;
    const int T = quarter * 32 + lane;  // TMEM lane = chunk row
    const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
    uint32_t r[32], r2[32];
    const float lg = kRet ? p.log2g[bh % max(p.ret_H, 1)] : 0.f;  // retention: log2 gamma
    for (int c = 0; c < nchunks; ++c) {
      const int s = c % kStages;
      const long tok = t_begin + (long)c * kC;
      bool w = mbar_wait(o_full, c & 1, abort_word, status, p.wait_ns) &&
               mbar_wait(&den_ready[c & 1], (c >> 1) & 1, abort_word, status, p.wait_ns);
      if (bar_or(kBarOut, 128, !w)) break;
      tc_fence_after();
      // normalizer, or (retention) the row's decay gamma^(T+1-C)
      const float inv = kRet ? exp2f((float)(T + 1 - min((long)kC, t_end - tok)) * lg) : 1.f / den_s[(c & 1) * kC + T];
      // normalised rows -> the V tile of this stage (free: P V has completed) as two
      // [128 x 32] fp32 swizzled boxes per half of the columns -> TMA stores.  Rows past
      // the sequence end are clipped by the store; the leading exact rows are rewritten later.
      // The second half is read from tensor memory before the first half's store drains,
      // so the accumulator is released as early as possible.
      uint8_t *stage_o = sm + Lay::V + s * kTile;
      for (int b = 0; b < 2; ++b) {
        tmem_ld32(tl + kColO + b * 32, r);
        uint8_t *box = stage_o + b * kBlk;
#pragma unroll
        for (int q = 0; q < 8; ++q) *reinterpret_cast<float4 *>(box + sw128_offset_f32(T, 4 * q)) = scale4(r + 4 * q, inv);
      }
      fence_async_smem();
      named_bar(kBarOut, 128);
      // A head's first chunk stores only rows 64..127: the exact pass writes rows 0..63
      // concurrently.  (Row 64 of a swizzled box starts 8 KB in, 1024-byte aligned.)
      const bool head_chunk = tok == 0 && p.n_exact > 0;
      if (T == 0 && !(head_chunk && p.N <= 64)) {
        if (head_chunk) {
          tma_store_3d(&p.to_tail, stage_o + 8192, 0, 64, bh);
          tma_store_3d(&p.to_tail, stage_o + kBlk + 8192, 32, 64, bh);
        } else {
          tma_store_3d(&p.to, stage_o, 0, (int)tok, bh);
          tma_store_3d(&p.to, stage_o + kBlk, 32, (int)tok, bh);
        }
      }
      if (T == 0) bulk_commit();
      tmem_ld32(tl + kColO + 64, r);
      tmem_ld32(tl + kColO + 96, r2);
      tc_fence_before();
      mbar_arrive(o_free);  // the O accumulator has been read
      if (T == 0) bulk_wait_read();
      named_bar(kBarOut, 128);  // the staging tile is free again
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        *reinterpret_cast<float4 *>(stage_o + sw128_offset_f32(T, 4 * q)) = scale4(r + 4 * q, inv);
        *reinterpret_cast<float4 *>(stage_o + kBlk + sw128_offset_f32(T, 4 * q)) = scale4(r2 + 4 * q, inv);
      }
      fence_async_smem();
      named_bar(kBarOut, 128);
      if (T == 0) {
        if (head_chunk) {
          if (p.N > 64) {
            tma_store_3d(&p.to_tail, stage_o + 8192, 64, 64, bh);
            tma_store_3d(&p.to_tail, stage_o + kBlk + 8192, 96, 64, bh);
          }
        } else {
          tma_store_3d(&p.to, stage_o, 64, (int)tok, bh);
          tma_store_3d(&p.to, stage_o + kBlk, 96, (int)tok, bh);
        }
        bulk_commit();
        bulk_wait_read();
        mbar_arrive(&v_empty[s]);  // the V tile may be reloaded
      }
    }
    if (T == 0) bulk_wait_all();  // output stores complete before the CTA exits
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, Lay::TmemCols);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() { return tensor_map_encoder(); }

// [BH][N][128] bf16 viewed as a 3-D tensor; boxes of 64 features x 128 tokens x 1 head.
bool make_map(CUtensorMap *m, const void *base, long BH, long N) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)N * kD * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)kC, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 output [BH][N][128]; boxes of 32 features x `rows` tokens x 1 head (128-byte rows).
bool make_out_map(CUtensorMap *m, void *base, long BH, long N, uint32_t rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)kD * 4, (cuuint64_t)N * kD * 4};
  cuuint32_t box[3] = {32, rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// One armed test injection (la_test_inject_missing_load): the chunk whose key
// load is left out and the wait limit in microseconds, packed as
// (chunk << 32) | wait_us; 0 when nothing is armed.  The next launch of the
// tensor-core causal pass takes it.
std::atomic<unsigned long long> g_inject{0};

template <int kMode>
cudaError_t launch_kernel(const TcParams &tp_in, dim3 grid, cudaStream_t stream, bool pdl) {
  constexpr bool kRet = kMode == kModeRetention;
  TcParams tp = tp_in;
  tp.wait_ns = kWaitNs;
  tp.skip_k_chunk = -1;
  if (const unsigned long long inj = g_inject.exchange(0)) {
    tp.skip_k_chunk = (int)(inj >> 32);
    tp.wait_ns = (inj & 0xffffffffull) * 1000ull;
  }
  const cudaError_t attr_err = ensure_smem_optin((const void *)causal_tc_kernel<kMode>, (int)Layout::Alloc);
  if (attr_err != cudaSuccess) return attr_err;
  LaunchTimer timer(kRet ? kKRetentionMain : kKCausalMain, stream);
  // pdl: may start while the previous kernel of the stream (the first pass) still runs
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Layout::Alloc;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, causal_tc_kernel<kMode>, tp);
  if (e == cudaSuccess) e = cudaGetLastError();
  timer.done(e);
  if (e == cudaSuccess) {
    count_launch();
  } else if (getenv("LA_DEBUG")) {
    cudaFuncAttributes fa;
    int blocks = -1;
    cudaFuncGetAttributes(&fa, causal_tc_kernel<kMode>);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, causal_tc_kernel<kMode>, kThreads, Layout::Alloc);
    fprintf(stderr,
            "linattn: causal_tc_kernel launch failed (%s): regs %d, max threads %d, static smem %zu, "
            "max dynamic smem %d, requested dynamic %u, threads %d, occupancy %d\n",
            cudaGetErrorString(e), fa.numRegs, fa.maxThreadsPerBlock, fa.sharedSizeBytes,
            fa.maxDynamicSharedSizeBytes, Layout::Alloc, kThreads, blocks);
    cudaGetLastError();
  }
  return e;
}

}  // namespace

// The passes of one call, all on the caller's stream, each allowed to start
// early (programmatic dependent launch) on the SMs its predecessor leaves free:
//   1. partial states of the earlier segments (first pass, when split);
//   2. the main tensor-core pass; segments that read partial states wait for
//      pass 1 to complete first;
//   3. the exact pass over each head's leading tokens, which reads nothing the
//      main pass writes and so runs beside it; its last CTA waits for pass 2,
//      so that the stream's next work follows all three.
// Retention (tp.ret_H > 0) runs passes 1 and 2 only: its segments past the
// first wait for pass 1, so pass 2 completes after it.
cudaError_t launch_passes(const Problem &p, const TcParams &tp, const float *S0, const float *z0, int mode) {
  cudaError_t e = cudaSuccess;
  const bool split = tp.nseg > 1, ret = mode == kModeRetention;
  if (split)
    e = launch_range_states(p, tp.seg_len, tp.fp_ranges, tp.fp_ctas, tp.fp_pieces_per_cta, tp.part_S, tp.part_z,
                            ret ? kKRetentionState : kKCausalState, ret ? tp.log2g : nullptr, tp.ret_H, mode);
  const dim3 grid((unsigned)tp.nseg, (unsigned)p.BH);
  if (e == cudaSuccess)
    e = ret                         ? launch_kernel<kModeRetention>(tp, grid, p.stream, split)
        : mode == kModeIdentity ? launch_kernel<kModeIdentity>(tp, grid, p.stream, split)
                                : launch_kernel<kModeElu>(tp, grid, p.stream, split);
  if (e == cudaSuccess && tp.n_exact > 0) e = launch_causal_exact_head(p, tp.n_exact, S0, z0, true);
  return e;
}

bool causal_tc_supported(const Problem &p) {
  const DeviceInfo &di = device_info(-1);
  return p.dt == LA_BF16 && p.dk == kD && p.dv == kD && di.cc_major == 10 && di.cc_minor == 3 &&
         p.N <= 0x7fffffffL && encode_fn() != nullptr;
}

// How one call cuts the work: G segments of seg_chunks chunks per head for the
// main pass, and (G > 1) a first pass over each head's G - 1 leading segments
// cut into `ctas` even runs of 64-token units, with one or two pieces a run;
// at most max_pieces pieces (the scratch that holds them).
struct Partition {
  long G = 1, seg_chunks = 0, ctas = 0, pieces_per_cta = 1;
  long pieces() const { return pieces_per_cta * ctas; }
};

// Segments per head forced by la_diag_force_segments (0: the planner's choice).
std::atomic<int> g_force_segments{0};

Partition plan_partition(const Problem &p, long sms, long max_pieces, bool allow_force = false) {
  Partition t;
  const long chunks = (p.N + kC - 1) / kC;
  // segments per head: enough CTAs to cover the SMs once, at least 4 chunks each
  t.G = std::max(1L, std::min(sms / p.BH, chunks / 4));
  const int forced = allow_force ? g_force_segments.load() : 0;
  if (forced > 0) t.G = std::min<long>(forced, chunks);
  t.seg_chunks = (chunks + t.G - 1) / t.G;
  t.G = (chunks + t.seg_chunks - 1) / t.seg_chunks;
  if (t.G > 1) {
    const long ranges = p.BH * (t.G - 1), L = t.seg_chunks * 2;  // first-pass segments, units each
    // runs that divide the segments (one piece each): the most CTAs within one wave
    long r = 1;
    for (long d = L; d >= 1; --d)
      if (L % d == 0 && ranges * d <= std::min(sms, max_pieces)) {
        r = d;
        break;
      }
    if (ranges * r * 5 >= sms * 4) {
      // they fill at least 80 % of the SMs: keep them (each main-pass segment then reads few pieces)
      t.ctas = ranges * r;
      t.pieces_per_cta = 1;
    } else {
      // otherwise one run per SM (fewer if the units run out), two pieces each; a run must not
      // exceed one segment
      t.ctas = std::min(std::min(sms, ranges * L), max_pieces / 2);
      t.pieces_per_cta = 2;
      if (t.ctas < ranges) t.ctas = 0;  // cannot be cut finely enough
    }
  }
  return t;
}

void set_first_pass(TcParams &tp, const Problem &p, const Partition &t) {
  tp.seg_len = (int)(t.seg_chunks * kC);
  tp.nseg = (int)t.G;
  tp.fp_ranges = (int)(t.G - 1);
  tp.fp_range_units = (int)(t.seg_chunks * 2);
  tp.fp_units = p.BH * (t.G - 1) * t.seg_chunks * 2;
  tp.fp_ctas = (int)t.ctas;
  tp.fp_pieces_per_cta = (int)t.pieces_per_cta;
}

// One call of the tensor-core path in one mode; retention decays head h by
// 2^log2g[h % ret_H].
cudaError_t launch_tc(const Problem &p, bool from_state, int mode, const float *log2g, int ret_H) {
  const bool ret = mode == kModeRetention;
  const DeviceInfo &di = device_info(-1);
  const long sms = std::max(1, di.sm_count);
  const Partition t = plan_partition(p, sms, 2 * sms, true);
  if (t.G > 1 && t.ctas == 0) return cudaErrorInvalidValue;  // not reached: BH * G <= SMs
  const long nparts = t.pieces();
  const size_t state_f = (size_t)kD * kD + kD;
  const size_t scratch_f = (size_t)nparts * state_f + (from_state ? (size_t)p.BH * state_f : 0);
  float *scratch = nullptr;
  cudaError_t e = cudaSuccess;
  if (scratch_f) {
    e = cudaMallocAsync(reinterpret_cast<void **>(&scratch), scratch_f * sizeof(float), p.stream);
    if (e != cudaSuccess) return e;
  }
  float *part_S = scratch;
  float *part_z = scratch ? part_S + (size_t)nparts * kD * kD : nullptr;
  const float *S0 = nullptr, *z0 = nullptr;
  if (from_state) {
    // the last segment overwrites the caller's state, so every reader uses a copy
    float *Sc = part_z + (size_t)nparts * kD;
    float *zc = Sc + (size_t)p.BH * kD * kD;
    e = cudaMemcpyAsync(Sc, p.S, sizeof(float) * p.BH * kD * kD, cudaMemcpyDeviceToDevice, p.stream);
    if (e == cudaSuccess && !ret)
      e = cudaMemcpyAsync(zc, p.z, sizeof(float) * p.BH * kD, cudaMemcpyDeviceToDevice, p.stream);
    if (e != cudaSuccess) {
      cudaFreeAsync(scratch, p.stream);
      return e;
    }
    S0 = Sc;
    z0 = ret ? nullptr : zc;
  }

  TcParams tp;
  memset(&tp, 0, sizeof tp);
  if (!make_map(&tp.tq, p.q, p.BH, p.N) || !make_map(&tp.tk, p.k, p.BH, p.N) ||
      !make_map(&tp.tv, p.v, p.BH, p.N) || !make_out_map(&tp.to, p.out, p.BH, p.N, kC) ||
      !make_out_map(&tp.to_tail, p.out, p.BH, p.N, 64)) {
    if (scratch) cudaFreeAsync(scratch, p.stream);
    return cudaErrorInvalidValue;
  }
  tp.out = p.out;
  tp.S_out = p.S;
  tp.z_out = p.z;
  tp.S0 = S0;
  tp.z0 = z0;
  tp.part_S = part_S;
  tp.part_z = part_z;
  tp.N = p.N;
  set_first_pass(tp, p, t);
  tp.n_exact = mode == kModeElu ? (int)std::min<long>(p.N, kExact) : 0;
  tp.eps = p.eps;
  tp.ret_H = ret ? ret_H : 0;
  for (int h = 0; ret && h < ret_H; ++h) tp.log2g[h] = log2g[h];

  e = launch_passes(p, tp, S0, z0, mode);
  if (scratch) {
    const cudaError_t f = cudaFreeAsync(scratch, p.stream);
    if (e == cudaSuccess) e = f;
  }
  return e;
}

void force_segments(int G) { g_force_segments.store(G); }

void arm_missing_load(int chunk, unsigned int wait_us) {
  g_inject.store(((unsigned long long)(unsigned)chunk << 32) | wait_us);
}

cudaError_t launch_causal_tc(const Problem &p, bool from_state) {
  return launch_tc(p, from_state, kModeElu, nullptr, 0);
}

cudaError_t launch_causal_features_tc(const Problem &p, bool from_state) {
  return launch_tc(p, from_state, kModeIdentity, nullptr, 0);
}

cudaError_t launch_retention_tc(const Problem &p, bool from_state, const float *log2g, int H) {
  if (!log2g || H < 1 || H > kMaxRetentionHeads) return cudaErrorInvalidValue;
  return launch_tc(p, from_state, kModeRetention, log2g, H);
}

// ---------------------------------------------------------------------------
// Allocation-free variant of the tensor-core causal pass (la_causal_noalloc).
// The partial states of the first pass live in this fixed array instead of a
// stream-ordered allocation; every device that loads the library keeps it
// until the process exits.  All calls share it and nothing in it needs to
// start at zero (every partial state is written before it is read), but calls
// that overlap on the GPU would race on it.
// ---------------------------------------------------------------------------
constexpr size_t kNoAllocScratchFloats = size_t(5) << 20;  // 20 MiB: the pieces of 158 first-pass CTAs
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchFloats];

namespace {
struct NoAllocScratch {
  float *ptr = nullptr;
  cudaError_t err = cudaErrorNotReady;
};

// Device address of the fixed scratch array, looked up once per device (with
// that device current, which the caller guarantees) on the first call that
// needs it.
NoAllocScratch noalloc_scratch(int dev) {
  static PerDeviceCache<int, NoAllocScratch> cache;
  return cache.get(dev, 0, [] {
    NoAllocScratch s;
    void *ptr = nullptr;
    s.err = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (s.err == cudaSuccess) s.ptr = static_cast<float *>(ptr);
    else cudaGetLastError();
    return s;
  });
}
}  // namespace

size_t noalloc_scratch_capacity_bytes() { return kNoAllocScratchFloats * sizeof(float); }

cudaError_t launch_causal_tc_noalloc(const Problem &p, int dev, bool *too_large) {
  *too_large = false;
  const DeviceInfo &di = device_info(dev);
  const long sms = std::max(1, di.sm_count);
  // the same partition as la_causal, with no more first-pass pieces than the fixed array holds
  const size_t state_f = (size_t)kD * kD + kD;
  const Partition t = plan_partition(p, sms, (long)(kNoAllocScratchFloats / state_f));
  if (t.G > 1 && t.ctas == 0) {
    *too_large = true;
    return cudaSuccess;
  }
  const long nparts = t.pieces();
  const size_t need = (size_t)nparts * state_f;
  float *part_S = nullptr, *part_z = nullptr;
  if (need) {
    const NoAllocScratch sc = noalloc_scratch(dev);
    if (sc.err != cudaSuccess) return sc.err;
    part_S = sc.ptr;
    part_z = part_S + (size_t)nparts * kD * kD;
  }
  TcParams tp;
  memset(&tp, 0, sizeof tp);
  if (!make_map(&tp.tq, p.q, p.BH, p.N) || !make_map(&tp.tk, p.k, p.BH, p.N) ||
      !make_map(&tp.tv, p.v, p.BH, p.N) || !make_out_map(&tp.to, p.out, p.BH, p.N, kC) ||
      !make_out_map(&tp.to_tail, p.out, p.BH, p.N, 64))
    return cudaErrorInvalidValue;
  tp.out = p.out;
  tp.S_out = p.S;
  tp.z_out = p.z;
  tp.part_S = part_S;
  tp.part_z = part_z;
  tp.N = p.N;
  set_first_pass(tp, p, t);
  tp.n_exact = (int)std::min<long>(p.N, kExact);
  tp.eps = p.eps;
  return launch_passes(p, tp, nullptr, nullptr, kModeElu);
}

cudaError_t read_and_clear_device_status(unsigned int *value) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(value, g_device_status, sizeof(unsigned int));
  if (e == cudaSuccess && *value) e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(unsigned int));
  return e;
}

}  // namespace la
