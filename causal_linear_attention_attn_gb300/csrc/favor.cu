// Positive random features ("Linear Attention Math", "Feature maps: elu+1 and
// positive random features"; "线性注意力从头到尾讲清楚" §9):
//   phi(x)_r = exp(w_r . x - |x|^2 / 2) / sqrt(m)
// for every row x of X ([rows, d]) and the m projections w_r (the rows of W).
//
// Tensor-core path (bf16, m = 128, d in {64, 128}): one persistent CTA per SM
// walks 128-row tiles.  Warp 0 issues the TMA loads (W once, X tiles
// double-buffered) and the MMA D = X W^T into one of two fp32 tensor-memory
// accumulators; two epilogue groups of four warps take alternate tiles, so
// that one group's exponentials overlap the next tile's MMA.  In a group
// every thread owns one row (its tensor-memory lane): it forms |x|^2 from the
// staged bf16 tile, applies the exponential, and writes bf16 features into
// the group's swizzled staging tile, which TMA stores copy out.  Other shapes
// and fp32 inputs take a plain CUDA-core kernel.  Every mbarrier wait is
// bounded; a wait that runs out raises the device status word and the CTA
// drains what it issued and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace la {

__device__ unsigned int g_favor_status;

namespace {
using namespace tc;

constexpr int kFavThreads = 288;         // warp 0: loads and MMAs; warps 1-4 and 5-8: two epilogue groups
constexpr int kFavM = 128;                 // features one tensor-core launch forms (m = 256: two launches)
constexpr uint32_t kBlk = 16384;           // [128 rows x 128 bytes], 128-byte swizzled
constexpr uint32_t kAbortMisaligned = 2u;  // status bit: shared memory base not 1024-aligned
constexpr uint32_t kBarGroup = 1;          // named barriers 1 and 2: the two epilogue groups

template <int D>
struct FavLayout {
  static constexpr uint32_t kTile = (D / 64) * kBlk;  // one [128 x D] bf16 tile
  static constexpr uint32_t W = 0;                    // the projections, [128 x D]
  static constexpr uint32_t X = W + kTile;            // two stages of X
  static constexpr uint32_t O = X + 2 * kTile;        // per group a [128 x 128] bf16 output staging tile
  static constexpr uint32_t Bars = O + 4 * kBlk;
  static constexpr uint32_t Misc = Bars + 12 * 8;
  static constexpr uint32_t Bytes = Misc + 16;
};

struct FavorParams {
  CUtensorMap tx, tw, to;  // X [1][rows][D], W [1][128][D] (128 of the m projections), out [1][rows][m], bf16, boxes 64 x 128
  int tiles;
  int col0;          // this launch's features are columns [col0, col0 + 128) of the m-wide output
  float inv_sqrt_m;  // 1 / sqrt(m) for the whole feature vector
};

// K-major operand (rows of 64 K-elements per 16 KB block): k-step ks covers K elements [16ks, 16ks+16).
__device__ __forceinline__ uint64_t kdesc(uint32_t tile, int ks) {
  return sw128_desc(tile + (ks >> 2) * kBlk + (ks & 3) * 32, 16, 1024);
}

// Tile i of this CTA uses X stage, accumulator and epilogue group i & 1; its
// barriers complete phase (i >> 1) & 1.
template <int D>
__global__ void __launch_bounds__(kFavThreads, 1) favor_tc_kernel(const __grid_constant__ FavorParams p) {
  using Lay = FavLayout<D>;
  extern __shared__ __align__(1024) uint8_t sm[];
  if (smem_u32(sm) & 1023u) {
    if (threadIdx.x == 0) atomicOr(&g_favor_status, kAbortMisaligned);
    return;
  }
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + Lay::Bars);
  // x_full: X landed; x_norm: the group has read its row norms; acc_full: MMA done (X read, D ready);
  // acc_free: the group has read D; w_full: W landed; drain: the last MMAs
  uint64_t *x_full = bars, *x_norm = bars + 2, *acc_full = bars + 4, *acc_free = bars + 6, *w_full = bars + 8,
           *drain = bars + 9;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + Lay::Misc);
  volatile uint32_t *abort_word = reinterpret_cast<volatile uint32_t *>(sm + Lay::Misc + 4);
  unsigned int *status = &g_favor_status;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n = blockIdx.x < p.tiles ? (p.tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  auto row0_of = [&](int i) { return ((int)blockIdx.x + i * (int)gridDim.x) * 128; };

  if (tid == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&x_full[b], 1);
      mbar_init(&x_norm[b], 128);
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_free[b], 128);
    }
    mbar_init(w_full, 1);
    mbar_init(drain, 1);
    *abort_word = 0;
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------- loads and MMAs (one thread) ----------------
    if (lane == 0 && n > 0) {
      prefetch_tmap(&p.tx);
      prefetch_tmap(&p.tw);
      mbar_arrive_expect_tx(w_full, Lay::kTile);
      for (int b = 0; b < D / 64; ++b) tma_load_3d(sm + Lay::W + b * kBlk, &p.tw, w_full, 64 * b, 0, 0);
      int loaded = 0, issued = 0;
      auto load_x = [&](int i) {
        const int s = i & 1;
        mbar_arrive_expect_tx(&x_full[s], Lay::kTile);
        for (int b = 0; b < D / 64; ++b)
          tma_load_3d(sm + Lay::X + s * Lay::kTile + b * kBlk, &p.tx, &x_full[s], 64 * b, row0_of(i), 0);
        loaded = i + 1;
      };
      load_x(0);
      if (n > 1) load_x(1);
      constexpr uint32_t kIdesc = idesc_bf16_f32(128, 128, 0, 0);
      const bool w_ok = mbar_wait(w_full, 0, abort_word, status);
      bool ok = w_ok;
      for (int i = 0; ok && i < n; ++i) {
        const int s = i & 1;
        const uint32_t ph = (i >> 1) & 1;
        ok = mbar_wait(&x_full[s], ph, abort_word, status);
        // the accumulator's previous tile (i - 2) has been read by its group
        if (ok && i >= 2) ok = mbar_wait(&acc_free[s], ph ^ 1, abort_word, status);
        if (!ok) break;
        tc_fence_after();
        const uint32_t xa = smem_u32(sm + Lay::X + s * Lay::kTile), wa = smem_u32(sm + Lay::W);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          mma_bf16(tmem + 128 * s, kdesc(xa, ks), kdesc(wa, ks), kIdesc, ks > 0);
        mma_commit(&acc_full[s]);
        issued = i + 1;
        // the stage takes tile i + 2 once this MMA and the group's norms have read it
        if (i + 2 < n) {
          ok = mbar_wait(&acc_full[s], ph, abort_word, status) && mbar_wait(&x_norm[s], ph, abort_word, status);
          if (ok) load_x(i + 2);
        }
      }
      // copies and MMAs still in flight land before the memory is released
      mma_commit(drain);
      wait_drain(drain, 0, status);
      for (int i = max(0, loaded - 2); i < loaded; ++i) wait_drain(&x_full[i & 1], (i >> 1) & 1, status);
      if (!w_ok) wait_drain(w_full, 0, status);
      (void)issued;
    }
  } else {
    // ---------------- two epilogue groups: group g takes tiles i with i & 1 == g ----------------
    const int g = (warp - 1) >> 2, gt = tid - 32 - 128 * g;  // gt: the row this thread owns
    const uint32_t lanes = (uint32_t)(32 * (warp & 3)) << 16;  // its tensor-memory lane quarter
    uint8_t *stage_o = sm + Lay::O + g * 2 * kBlk;
    const float inv_sqrt_m = p.inv_sqrt_m;
    const int row = 32 * (warp & 3) + lane;  // tensor-memory lane = tile row
    (void)gt;
    for (int i = g; i < n; i += 2) {
      const uint32_t ph = (i >> 1) & 1;
      const uint8_t *xs = sm + Lay::X + g * Lay::kTile;
      bool ok = mbar_wait(&x_full[g], ph, abort_word, status);
      if (bar_or(kBarGroup + g, 128, !ok)) break;
      float nrm = 0.f;
#pragma unroll
      for (int b = 0; b < D / 64; ++b)
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 w = *reinterpret_cast<const uint4 *>(xs + b * kBlk + sw128_offset(row, 8 * c));
          const uint32_t e[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float lo = __uint_as_float(e[j] << 16), hi = __uint_as_float(e[j] & 0xffff0000u);
            nrm = fmaf(lo, lo, nrm);
            nrm = fmaf(hi, hi, nrm);
          }
        }
      mbar_arrive(&x_norm[g]);
      ok = mbar_wait(&acc_full[g], ph, abort_word, status);
      if (row == 0) bulk_wait_read();  // this group's previous stores have read its staging tile
      if (bar_or(kBarGroup + g, 128, !ok)) break;
      tc_fence_after();
#pragma unroll 1
      for (int cb = 0; cb < 4; ++cb) {
        uint32_t r[32];
        tmem_ld32(tmem + 128 * g + lanes + cb * 32, r);
        uint8_t *blk = stage_o + (cb >> 1) * kBlk;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t o[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float a = __expf(__uint_as_float(r[8 * q + 2 * j]) - 0.5f * nrm) * inv_sqrt_m;
            const float b = __expf(__uint_as_float(r[8 * q + 2 * j + 1]) - 0.5f * nrm) * inv_sqrt_m;
            o[j] = pack_bf16(a, b);
          }
          *reinterpret_cast<uint4 *>(blk + sw128_offset(row, (cb & 1) * 32 + 8 * q)) = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
      tc_fence_before();
      mbar_arrive(&acc_free[g]);  // the accumulator may take tile i + 2
      fence_async_smem();
      named_bar(kBarGroup + g, 128);
      if (row == 0) {
        tma_store_3d(&p.to, stage_o, p.col0, row0_of(i), 0);
        tma_store_3d(&p.to, stage_o + kBlk, p.col0 + 64, row0_of(i), 0);
        bulk_commit();
      }
    }
    if (row == 0) bulk_wait_all();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// One row per block: the row in shared memory, its norm by a block reduction,
// then every feature as a plain dot product with its projection.
template <typename Tin>
__global__ void __launch_bounds__(128) favor_simt_kernel(const Tin *__restrict__ X, const Tin *__restrict__ W,
                                                         Tin *__restrict__ out, int d, int m) {
  extern __shared__ float xs[];
  __shared__ float part[4];
  const long row = blockIdx.x;
  const int tid = threadIdx.x;
  float nrm = 0.f;
  for (int i = tid; i < d; i += 128) {
    const float x = ldf(X + row * d + i);
    xs[i] = x;
    nrm = fmaf(x, x, nrm);
  }
  nrm = warp_sum(nrm);
  if ((tid & 31) == 0) part[tid >> 5] = nrm;
  __syncthreads();
  nrm = part[0] + part[1] + part[2] + part[3];
  const float inv_sqrt_m = 1.f / sqrtf((float)m);
  for (int f = tid; f < m; f += 128) {
    float wx = 0.f;
    for (int i = 0; i < d; ++i) wx = fmaf(ldf(W + (long)f * d + i), xs[i], wx);
    const float y = expf(wx - 0.5f * nrm) * inv_sqrt_m;
    if constexpr (sizeof(Tin) == 4)
      out[row * m + f] = y;
    else
      out[row * m + f] = __float2bfloat16_rn(y);
  }
}

bool make_map2(CUtensorMap *map, const void *base, long rows, int cols) {
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, 1};
  cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)rows * cols * 2};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// m = 128 h features: one launch per block of 128 projections, each writing its columns of the
// m-wide rows (X is read once per launch).
template <int D>
cudaError_t launch_tc(const void *X, const void *W, void *out, long rows, int m, cudaStream_t stream) {
  using Lay = FavLayout<D>;
  const cudaError_t attr = ensure_smem_optin((const void *)favor_tc_kernel<D>, (int)Lay::Bytes);
  if (attr != cudaSuccess) return attr;
  const int sms = std::max(1, device_info(-1).sm_count);
  for (int col0 = 0; col0 < m; col0 += kFavM) {
    FavorParams p;
    const void *Wb = static_cast<const __nv_bfloat16 *>(W) + (long)col0 * D;
    if (!make_map2(&p.tx, X, rows, D) || !make_map2(&p.tw, Wb, kFavM, D) || !make_map2(&p.to, out, rows, m))
      return cudaErrorInvalidValue;
    p.tiles = (int)((rows + 127) / 128);
    p.col0 = col0;
    p.inv_sqrt_m = (float)(1.0 / std::sqrt((double)m));
    LaunchTimer timer(kKFavor, stream);
    favor_tc_kernel<D><<<std::min(p.tiles, sms), kFavThreads, Lay::Bytes, stream>>>(p);
    const cudaError_t e = cudaGetLastError();
    timer.done(e);
    if (e != cudaSuccess) return e;
    count_launch();
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_favor_features(const void *X, const void *W, void *out, long rows, int d, int m, la_dtype dt,
                                  cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  const DeviceInfo &di = device_info(-1);
  const bool tc = dt == LA_BF16 && (m == kFavM || m == 2 * kFavM) && (d == 64 || d == 128) && rows <= 0x7fffff80L &&
                  di.cc_major == 10 && di.cc_minor == 3 && tensor_map_encoder() != nullptr;
  if (tc) return d == 64 ? launch_tc<64>(X, W, out, rows, m, stream) : launch_tc<128>(X, W, out, rows, m, stream);
  LaunchTimer timer(kKFavor, stream);
  if (dt == LA_F32)
    favor_simt_kernel<float><<<(unsigned)rows, 128, sizeof(float) * d, stream>>>(
        (const float *)X, (const float *)W, (float *)out, d, m);
  else
    favor_simt_kernel<__nv_bfloat16><<<(unsigned)rows, 128, sizeof(float) * d, stream>>>(
        (const __nv_bfloat16 *)X, (const __nv_bfloat16 *)W, (__nv_bfloat16 *)out, d, m);
  const cudaError_t e = cudaGetLastError();
  timer.done(e);
  if (e == cudaSuccess) count_launch();
  return e;
}

cudaError_t read_and_clear_favor_status(unsigned int *value) {
  const unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(value, g_favor_status, sizeof(unsigned int));
  if (e == cudaSuccess && *value) e = cudaMemcpyToSymbol(g_favor_status, &zero, sizeof(unsigned int));
  return e;
}

}  // namespace la
