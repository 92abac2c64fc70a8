// Host-side launcher declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "linattn.h"

namespace la {

// One call's problem, heads flattened to BH = B * H.  Pointers are device
// pointers as documented in linattn.h.
struct Problem {
  const void *q, *k, *v;
  float *out, *S, *z;
  int BH;
  long N;
  int dk, dv;
  float eps;
  la_dtype dt;
  cudaStream_t stream;
};

// Gradient of the causal prefill: the problem's q, k, v, eps and sizes, the
// upstream gradient of the output, the forward's initial state (nullable)
// and the gradient of its final state (nullable); the gradients of q, k, v
// and (nullable) of the initial state are written.  All device pointers.
struct BackwardProblem {
  Problem p;
  const float *dout, *S0, *z0, *dS, *dz;
  float *dq, *dk, *dv, *dS0, *dz0;
};
cudaError_t launch_causal_backward(const BackwardProblem &b);
// The same gradient on the tensor cores (bf16 inputs, d_k = d_v = 128, N >= 1, sm_103,
// q, k, dq, dk, dv 32-byte aligned).
bool backward_tc_supported(const BackwardProblem &b);
cudaError_t launch_causal_backward_tc(const BackwardProblem &b);
cudaError_t read_and_clear_backward_status(unsigned int *value);

// Exact fp32 CUDA-core chunked causal pass.  Processes tokens [0, n_proc) of
// every head.  from_state: start from the caller's S, z instead of zero.
// write_state: store the final S, z.
// identity: q and k are given features (no phi).
cudaError_t launch_causal_simt(const Problem &p, long n_proc, bool from_state, bool write_state,
                               bool identity = false);

// Exact fp32 pass over tokens [0, n_exact) of every head (outputs only),
// starting from (S0, z0) when given (device pointers), else from zero.  With
// pdl it may start while the previous kernel of the stream runs (it must not
// read that kernel's results); its last CTA waits for that kernel, so the
// stream's later work still follows both.
cudaError_t launch_causal_exact_head(const Problem &p, long n_exact, const float *S0, const float *z0, bool pdl);

// Tensor-core chunked causal path (bf16, d_k = d_v = 128, sm_103).
bool causal_tc_supported(const Problem &p);
cudaError_t launch_causal_tc(const Problem &p, bool from_state);
// Retention on the same path: head bh decays by 2^log2g[bh % H] (host array, H <= 128).
cudaError_t launch_retention_tc(const Problem &p, bool from_state, const float *log2g, int H);
// Normalized causal attention on given features (q, k are phi(q), phi(k)).
cudaError_t launch_causal_features_tc(const Problem &p, bool from_state);

// Positive random features of `rows` rows of X ([rows, d]) for W ([m, d]) into out ([rows, m]),
// all of dtype dt; the tensor cores take bf16 with m = 128 and d in {64, 128}.
cudaError_t launch_favor_features(const void *X, const void *W, void *out, long rows, int d, int m, la_dtype dt,
                                  cudaStream_t stream);
cudaError_t read_and_clear_favor_status(unsigned int *value);

// Allocation-free tensor-core causal pass from the zero state: the first
// pass's partial states use a fixed device array instead of an allocation.
// Sets *too_large (and launches nothing) if they would not fit.
cudaError_t launch_causal_tc_noalloc(const Problem &p, int dev, bool *too_large);
size_t noalloc_scratch_capacity_bytes();

// cuTensorMapEncodeTiled, looked up once through the runtime (the library
// does not link libcuda); nullptr if the driver does not provide it.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// Tensor-core global form (bf16, d_k = d_v in {64, 128}): state build, then read (for d = 64
// with enough heads to fill the SMs, both in one kernel, a CTA per head).
bool global_tc_supported(const Problem &p);
cudaError_t launch_global_tc(const Problem &p);
cudaError_t read_and_clear_global_tc_status(unsigned int *value);

// First pass of the split causal form on the tensor cores (bf16, d_k = d_v = 128).
// Each head's first ranges_per_head ranges of range_tokens tokens (range s of
// head h is r = h * ranges_per_head + s), all heads one after another, are cut
// evenly into `ctas` runs of 64-token units, one per CTA; a run must be at most
// one range long (ctas >= BH * ranges_per_head), so it spans at most two ranges.
// CTA c writes the sums of phi(k) v^T and phi(k) over the part of its run in its
// first range to piece 2c and over the rest to piece 2c + 1 (zeros if none):
// piece_S[piece][128][128], piece_z[piece][128].  range_tokens % 64 == 0.  With
// pieces_per_cta == 1 the runs must divide the ranges evenly; CTA c then writes
// piece c only.
// Retention: per-head decays gamma_h carried in launch parameters, at most this many heads.
constexpr int kMaxRetentionHeads = 128;

// What the tensor-core causal passes compute: normalized attention with phi = ELU + 1, retention
// (decay, no denominator), or normalized attention on features the caller has already applied.
enum TcMode : int { kModeElu = 0, kModeRetention = 1, kModeIdentity = 2 };

// log2g (host array of ret_H values, or null): retention weights instead of phi and key sums.
cudaError_t launch_range_states(const Problem &p, long range_tokens, int ranges_per_head, int ctas, int pieces_per_cta,
                                float *piece_S, float *piece_z, int kernel_id, const float *log2g = nullptr,
                                int ret_H = 0, int mode = kModeElu);

// Testing: the next launch of the tensor-core causal pass leaves out the key
// load of `chunk` in its first CTA and gives every mbarrier wait wait_us
// microseconds (see la_test_inject_missing_load).
void arm_missing_load(int chunk, unsigned int wait_us);

// Diagnostics: segments per head of the tensor-core causal passes (0: planner).
void force_segments(int G);

// Read and clear the device status word (bounded-wait timeouts).
cudaError_t read_and_clear_device_status(unsigned int *value);

// Global form: state build (S, z are zeroed and accumulated) then the read.
// identity: q and k are given features (no phi).
cudaError_t launch_global_simt(const Problem &p, bool identity = false);

// One decode step, S and z in place.
cudaError_t launch_decode(const Problem &p);
// Retention decode step: S = gamma[bh % H] S + k v^T, out = q^T S (host gamma array, H <= 128; no z).
cudaError_t launch_retention_decode(const Problem &p, const float *gamma, int H);
// Retention prefill on CUDA cores, exact fp32, any supported dtype and head size, gamma in [0, 1]
// (host array, head bh decays by gamma[bh % H], H <= 128).
cudaError_t launch_retention_simt(const Problem &p, bool from_state, const float *gamma, int H);

// Count one successful kernel launch (reported by la_kernel_launches).
void count_launch(unsigned n = 1);

// Kernel ids of the device-time diagnostics (same values as la_kernel).
enum KernelId : int {
  kKCausalMain = 0,
  kKCausalState = 1,
  kKExactHead = 2,
  kKCausalSimt = 3,
  kKGlobalState = 4,
  kKGlobalRead = 5,
  kKDecode = 6,
  kKRetentionMain = 7,
  kKRetentionState = 8,
  kKRetentionDecode = 9,
  kKBackward = 10,
  kKFavor = 11,
  kKGlobalFused = 12,
  kKNumKernels = 13
};

// While profiling is on (la_profile_enable), brackets one launch with a CUDA
// event pair on its stream; construct it just before the launch and call
// done() with the launch's error just after.  Costs nothing when off.
class LaunchTimer {
 public:
  LaunchTimer(int kernel, cudaStream_t stream);
  void done(cudaError_t launch_error);

 private:
  int kernel_;
  cudaStream_t stream_;
  cudaEvent_t start_ = nullptr;
};

// Opt a kernel in to `bytes` of dynamic shared memory on the current device.
// The attribute lives in each device's context, so it is set once per
// (device, kernel, size) and the result is remembered for that device only.
cudaError_t ensure_smem_optin(const void *kernel, int bytes);

// Per-device attributes, read once per device (dev < 0: the current device;
// all zero if there is none).
struct DeviceInfo {
  int sm_count = 0;
  int cc_major = 0, cc_minor = 0;
  int max_smem_optin = 0;
};
DeviceInfo device_info(int dev);

}  // namespace la
