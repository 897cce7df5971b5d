// Internal interface between the host library (zero_host.cpp) and the CUDA
// kernels (zero_kernels.cu). Not part of the public C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "zero_gb300.h"

namespace zk {

constexpr int kMaxRanks = ZERO_MAX_RANKS;

// A contiguous index range [lo, lo + head + nvec*V + tail) split into a scalar
// head (up to the first index where every buffer is 16-byte aligned), nvec
// V-element vector units, and a scalar tail. When the buffers do not share a
// 16-byte phase the whole range is the head (nvec = tail = 0).
struct Split {
  int64_t lo;
  int64_t head;
  int64_t nvec;
  int64_t tail;
};

// Per-step float32 constants, formed in double on the host and rounded once.
struct AdamConsts {
  float decay;  // 1 - lr*wd
  float b1;     // beta1
  float omb1;   // 1 - beta1
  float b2;     // beta2
  float omb2;   // 1 - beta2
  float step;   // lr / (1 - beta1^t)
  float bc2s;   // sqrt(1 - beta2^t)
  float eps;
};

// Per-step float32 constants of momentum SGD, formed in double on the host and
// rounded once, with its switches.
struct SgdConsts {
  float lr;
  float wd;          // coupled decay g += wd*p, applied when wd_on
  float mu;          // momentum
  float omd;         // 1 - dampening
  int32_t wd_on;
  int32_t first;     // t == 1: the buffer starts as the gradient
  int32_t nesterov;
};

// Kernel argument block of the fused step (passed by value as a
// __grid_constant__ parameter; about 1.7 KB).
struct StepArgs {
  const void* grads[kMaxRanks];  // N gradient buffers (float or bf16)
  void* reps[kMaxRanks];         // N parameter replicas (float or bf16)
  int64_t bounds[kMaxRanks + 1]; // shard offsets a_0..a_N (owner lookup)
  float* m;                      // flat fp32 state, global index order
  float* v;
  float* master;                 // mixed precision only
  Split sp;
  int32_t N;
  float fN;                      // (float)N
  AdamConsts c;                  // AdamW steps
  SgdConsts sgd;                 // momentum-SGD steps (the buffer is m)
  // Multiplier of the mean gradient: gscale, times the clip coefficient
  // min(1, max_norm / (gscale * sqrt(*norm_sq) + 1e-6)) when norm_sq is set
  // (formed on the device, in double, rounded to float once).
  // Device scalar, or NULL (no clipping). When the launch is a programmatic
  // dependent, the kernel waits for the kernel before it (the norm's total)
  // before reading it.
  const double* norm_sq;
  double gscale;
  double max_norm;
  // The multiplier when there is no clipping (norm_sq NULL): float(gscale),
  // formed on the host -- the device's double pipe is slow, and a one-pass
  // grid has millions of threads.
  float gm;
  // Stage 3: write the new parameters only into the owner's replica, over the
  // owner's shard; the other replicas' elements are left untouched.
  int32_t owner_only;
  // Launch as a programmatic dependent of the previous kernel on the stream:
  // a later bucket of the same step (disjoint indices), or a clipped step
  // after the kernel that writes norm_sq.
  int32_t dependent;
  // A clipped step whose call formed the norm itself: the multiplier, formed
  // from norm_sq by the norm's total kernel (NormArgs::gm_out), read instead of
  // forming it again in every block. NULL otherwise.
  const float* gm_dev;
};

// Squared global norm of the mean gradient, as fixed-size partial sums.
constexpr int64_t kNormChunk = 32768;  // elements per partial sum

struct NormArgs {
  const void* grads[kMaxRanks];
  Split sp;          // the whole range [0, n)
  int32_t N;
  float fN;
  // Elements per partial sum, kNormChunk. Passed at run time: the kernel with
  // this as a compile-time constant measured 3-7 % slower (and chunks of
  // 2,048-16,384 elements, for a more even spread over the SMs, slower still).
  int64_t chunk;
  int64_t nchunks;   // vector chunks (chunk / V units each); partial nchunks = scalars
  // The partials this launch computes: [c_begin, c_end) within [0, nchunks]
  // (index nchunks is the scalar head and tail). The whole pass is
  // [0, nchunks + 1); the host-input step launches the chunks of each piece of
  // the gradient as soon as it has arrived.
  int64_t c_begin, c_end;
  double* partials;  // nchunks + 1 doubles
  double* out;       // device scalar receiving the sum of the partials
  // A clipped step chained to this norm: the total kernel also forms the
  // step's gradient multiplier from the total (gscale, max_norm as in
  // StepArgs) into *gm_out, the float slot after the partials in the caller's
  // scratch. NULL: the norm alone.
  float* gm_out;
  double gscale, max_norm;
};

// The caller's norm scratch: the nchunks + 1 partial sums, then one double
// slot holding the chained step's multiplier (a float in its first 4 bytes).
constexpr int64_t kNormScratchExtra = 2;

struct AllreduceArgs {
  void* grads[kMaxRanks];
  Split sp;
  int32_t N;
  float fN;
};

// Stage-3 all-gather: copy each shard [bounds[r], bounds[r+1]) of replica r
// into every other replica, over the range of sp.
struct GatherArgs {
  void* reps[kMaxRanks];
  int64_t bounds[kMaxRanks + 1];
  Split sp;
  int32_t N;
};

struct InitArgs {
  float* m;
  float* v;
  float* master;       // NULL in fp32
  const float* init;   // NULL in fp32
  Split sp;
};

// The optimizer a fused step runs. Each keeps some fp32 state streams per
// parameter besides the parameter (or master): AdamW m and v, momentum SGD
// its buffer (in m), plain SGD none.
enum class Opt : int { AdamW = 0, SgdMomentum = 1, Sgd = 2 };

// Launchers (zero_kernels.cu). Each returns the launch status.
cudaError_t launch_step(const StepArgs& a, bool mixed, Opt opt, cudaStream_t s);
cudaError_t launch_allreduce(const AllreduceArgs& a, bool bf16, cudaStream_t s);
cudaError_t launch_init(const InitArgs& a, cudaStream_t s);
cudaError_t launch_gather(const GatherArgs& a, bool bf16, cudaStream_t s);
// Partial sums then their fixed-order total (two launches, deterministic).
cudaError_t launch_norm(const NormArgs& a, bool bf16, cudaStream_t s);
// The partials [a.c_begin, a.c_end) only (one launch; its blocks let a
// programmatic dependent start early), and the fixed-order total only (one
// block, launched as a programmatic dependent of the kernel before it, which
// it waits for before reading the partials; it lets its own dependent start).
cudaError_t launch_norm_partials(const NormArgs& a, bool bf16, cudaStream_t s);
cudaError_t launch_norm_total(const NormArgs& a, cudaStream_t s);

// Capacity of the library's own partial-sum array (zero_grad_norm_sq_noalloc),
// and the device address of that array on the current device (looked up on
// first use per device).
constexpr int64_t kNoAllocPartials = 65536;
cudaError_t noalloc_partials(double** ptr);


}  // namespace zk
