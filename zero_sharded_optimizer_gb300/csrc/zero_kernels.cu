// CUDA kernels (sm_103a) of the ZeRO step over N simulated ranks in one HBM.
//
// The fused step does, per index j and in one pass over memory:
//   reduce-scatter-mean  g = (sum_r g_r[j]) / N             (rank order 0..N-1)
//   AdamW on the shard   p, m, v -> p', m', v'              (owner's state)
//   all-gather           replica_r[j] = p' for every r      (bf16: RNE(p'))
// ("ZeRO-Sharded Adam Step", section "The step"; "Data parallelism and ZeRO
// stages 1 to 3", section 2, stages 1 and 2). The state is flat in global
// index order, so the shard structure only decides whose replica holds the
// authoritative fp32 parameter (the owner's) -- never the arithmetic. Variants:
// momentum SGD in place of AdamW, and the stage-3 owner-only step (no
// all-gather; gather_kernel brings the replicas back).
//
// The step moves 8N+20 bytes per parameter in fp32 (4N+24 in mixed precision)
// and does ~20 flops per parameter: it is bound by HBM bandwidth. One kernel
// runs it, zero_step_kernel: register streaming with 16-byte vector
// loads/stores, one V-element unit per thread (V = 4 fp32, V = 8 mixed), every
// load of a unit issued before any arithmetic, streaming cache hints
// (ld/st .cs), and a scalar head/tail for ranges whose ends are not on a unit
// boundary. Its grid is one pass over the units: a block per stretch of units,
// launched in waves, each block exiting after its stretch, so the blocks that
// run at one time work on one contiguous window of memory. This measured 3-6 %
// faster than a persistent bulk-copy (TMA) pipeline through shared memory and
// than a persistent grid-stride grid of the same kernel; fp32 AdamW with one
// rank alone keeps the grid-stride grid, and fp32 SGD with one rank takes two
// units per thread. The stage-3 gather and the DDP mean are register
// streaming in one pass too. Bucket launches of one step are programmatic
// dependents of the one before (their ramp and tail overlap); every kernel
// still completes in stream order. No kernel waits on another block or on a
// copy, so nothing waits on the device.
// Every kernel uses explicitly rounded IEEE fp32 intrinsics (__fadd_rn,
// __fmul_rn, __fdiv_rn, __fsqrt_rn): no contraction, so the result is
// independent of compiler scheduling and bit-reproducible. No tensor cores:
// there is no contraction in this step.

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cstring>
#include <mutex>
#include <type_traits>

#include "zero_internal.h"

namespace zk {
namespace {

constexpr int kThreads = 256;

// ----------------------------------------------------------- memory helpers --

__device__ __forceinline__ float4 ld4(const float* p) {
  return __ldcs(reinterpret_cast<const float4*>(p));
}
__device__ __forceinline__ uint4 ld8h(const uint16_t* p) {
  return __ldcs(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ void st4(float* p, float4 x) {
  __stcs(reinterpret_cast<float4*>(p), x);
}
__device__ __forceinline__ void st8h(uint16_t* p, uint4 x) {
  __stcs(reinterpret_cast<uint4*>(p), x);
}

// bf16 <-> fp32. Widening is exact (the bf16 bits are the top half of the
// fp32 bits); narrowing uses CUDA's round-to-nearest-even conversion.
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf_one(uint16_t h) { return __uint_as_float(uint32_t(h) << 16); }
__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint16_t to_bf(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

__device__ __forceinline__ void unpack8(uint4 w, float (&f)[8]) {
  f[0] = bf_lo(w.x); f[1] = bf_hi(w.x);
  f[2] = bf_lo(w.y); f[3] = bf_hi(w.y);
  f[4] = bf_lo(w.z); f[5] = bf_hi(w.z);
  f[6] = bf_lo(w.w); f[7] = bf_hi(w.w);
}
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  return make_uint4(pack_bf2(f[0], f[1]), pack_bf2(f[2], f[3]), pack_bf2(f[4], f[5]),
                    pack_bf2(f[6], f[7]));
}
__device__ __forceinline__ float4 unpack4(uint2 w) {
  return make_float4(bf_lo(w.x), bf_hi(w.x), bf_lo(w.y), bf_hi(w.y));
}
__device__ __forceinline__ uint2 pack4(float4 f) {
  return make_uint2(pack_bf2(f.x, f.y), pack_bf2(f.z, f.w));
}

// Programmatic dependent launch: let the next kernel on the stream start
// (once every CTA here has said so), and wait for the kernel before this one
// to complete with its memory visible (a no-op when this kernel was launched
// without the attribute).
__device__ __forceinline__ void pdl_allow_next() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_previous() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// The fixed-order total of `count` non-negative doubles (partial sums of
// squares), the same bits on every call: thread t < 256 adds p[t], p[t + 256],
// ... in that order, eight loads in flight (past the end they read as +0.0,
// which leaves the non-negative running sum unchanged); each warp folds its 32
// sums by one fixed shuffle tree; thread 0 adds the warp sums in warp order,
// starting from zero. Called by every thread of a block of 256; the result is
// valid in thread 0.
__device__ __forceinline__ double fixed_order_total(const double* p, int64_t count) {
  __shared__ double warp_sums[32];
  const int lt = threadIdx.x;
  double acc = 0.0;
  for (int64_t c = lt; c < count; c += 8 * 256) {
    double x[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) x[u] = c + u * 256 < count ? p[c + u * 256] : 0.0;
#pragma unroll
    for (int u = 0; u < 8; ++u) acc += x[u];
  }
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_down_sync(0xffffffffu, acc, off);
  if ((lt & 31) == 0) warp_sums[lt >> 5] = acc;
  __syncthreads();
  double t = 0.0;
  if (lt == 0)
    for (int w = 0; w < int(blockDim.x / 32); ++w) t += warp_sums[w];
  return t;
}

// ----------------------------------------------------------------- the math --

// Divide the rank-ordered sum by N. For a power-of-two N the product with 1/N
// is the same correctly rounded value as the quotient, so it is used instead.
template <int NR>
__device__ __forceinline__ float mean_of(float s, float fN) {
  if constexpr (NR > 0 && (NR & (NR - 1)) == 0) {
    return __fmul_rn(s, 1.0f / float(NR));
  } else {
    return __fdiv_rn(s, fN);
  }
}

// Correctly rounded sqrt(v) for v >= 0, equal to __fsqrt_rn(v), with zero and
// subnormal inputs answered through exact identities so the square root itself
// only ever sees normal numbers: sqrt(+-0) = +-0, and for subnormal v
// sqrt(v) = sqrt(v * 2^24) * 2^-12 (both scalings by powers of two are exact
// and commute with rounding because every intermediate is normal). Gradients
// that are exactly zero keep m and v at zero, or decaying through the
// subnormal range; this keeps those elements on the same instruction path as
// their neighbours in the warp.
__device__ __forceinline__ float sqrt_nonneg(float v) {
  const bool normal = v >= 0x1p-126f;  // also +inf
  const bool sub = v > 0.0f && !normal;
  const float r = __fsqrt_rn(normal ? v : (sub ? __fmul_rn(v, 0x1p24f) : 1.0f));
  if (normal) return r;
  if (sub) return __fmul_rn(r, 0x1p-12f);
  if (v == 0.0f) return v;
  return __fsqrt_rn(v);  // negative or NaN: the IEEE result
}

// Correctly rounded a / b for b > 0, equal to __fdiv_rn(a, b), with zero and
// subnormal numerators answered through exact identities: +-0 / b = +-0, and
// for subnormal a with a normal quotient a / b = ((a * 2^24) / b) * 2^-24.
__device__ __forceinline__ float div_by_pos(float a, float b) {
  const float aa = fabsf(a);
  const bool zero = aa == 0.0f;
  const bool sub = aa > 0.0f && aa < 0x1p-126f;
  const float q = __fdiv_rn(zero ? 1.0f : (sub ? __fmul_rn(a, 0x1p24f) : a), b);
  if (!(b > 0.0f)) return __fdiv_rn(a, b);  // outside the expected domain: IEEE as is
  if (zero) return a;
  if (sub) return fabsf(q) >= 0x1p-101f ? __fmul_rn(q, 0x1p-24f) : __fdiv_rn(a, b);
  return q;
}

// One AdamW element: decoupled decay, moments, bias-corrected update.
__device__ __forceinline__ void adam1(const AdamConsts& c, float g, float& p, float& m,
                                      float& v) {
  p = __fmul_rn(p, c.decay);
  m = __fadd_rn(__fmul_rn(c.b1, m), __fmul_rn(c.omb1, g));
  v = __fadd_rn(__fmul_rn(c.b2, v), __fmul_rn(c.omb2, __fmul_rn(g, g)));
  const float d = __fadd_rn(div_by_pos(sqrt_nonneg(v), c.bc2s), c.eps);
  p = __fsub_rn(p, __fmul_rn(c.step, div_by_pos(m, d)));
}

template <int NR>
__device__ __forceinline__ int ranks(const StepArgs& P) {
  return NR > 0 ? NR : P.N;
}

// Multiplier of the mean gradient when clipping: the accumulation factor
// gscale times the clip coefficient
// min(1, max_norm / (gscale * sqrt(norm_sq) + 1e-6)). Formed in double with
// separately rounded operations (no contraction), rounded to float once.
__device__ __forceinline__ float clip_multiplier(double gscale, double max_norm, double norm_sq) {
  const double denom = __dadd_rn(__dmul_rn(gscale, __dsqrt_rn(norm_sq)), 1e-6);
  const double c = fmin(1.0, __ddiv_rn(max_norm, denom));
  return __double2float_rn(__dmul_rn(gscale, c));
}

// The multiplier of a block's threads. Without clipping: the host's
// float(gscale) (the same value: gscale * 1 rounded to float once). A clipped
// step chained to its norm: the multiplier the norm's total kernel formed,
// read from memory by every thread (no barrier, so the unit loads are not held
// behind it). Otherwise thread 0 forms it from the squared norm in double and
// the block shares it: the double pipe is slow, so once per block, not per
// thread. Every thread of the block must call it.
__device__ __forceinline__ float block_grad_multiplier(const StepArgs& P) {
  if (!P.norm_sq) return P.gm;
  if (P.gm_dev) return *P.gm_dev;
  __shared__ float shared_gm;
  if (threadIdx.x == 0) shared_gm = clip_multiplier(P.gscale, P.max_norm, *P.norm_sq);
  __syncthreads();
  return shared_gm;
}

// The mean of the rank-ordered sum, times the gradient multiplier.
template <int NR>
__device__ __forceinline__ float scaled_mean(float s, const StepArgs& P, float gm) {
  return __fmul_rn(mean_of<NR>(s, P.fN), gm);
}

// Owner of index j, advanced monotonically from `owner` (j never decreases
// along one thread's iterations). bounds[N] = n > j stops the scan.
__device__ __forceinline__ int advance_owner(const StepArgs& P, int owner, int64_t j) {
  while (j >= P.bounds[owner + 1]) ++owner;
  return owner;
}

// ------------------------------------------------------ the optimizer update --

// fp32 state streams per parameter besides the parameter itself; arrays are
// sized at least 1.
template <Opt O>
constexpr int kStates = O == Opt::AdamW ? 2 : (O == Opt::SgdMomentum ? 1 : 0);
template <Opt O>
constexpr int kSA = kStates<O> > 0 ? kStates<O> : 1;

// State stream k: m (AdamW's first moment, or the SGD momentum buffer), v.
__device__ __forceinline__ float* state_ptr(const StepArgs& P, int k) {
  return k == 0 ? P.m : P.v;
}

// One momentum-SGD element (torch.optim.SGD semantics): coupled decay
// g += wd*p; the buffer is g at the first step, else mu*buf + (1-dampening)*g;
// the direction is the buffer, or g + mu*buf with Nesterov (plain SGD: g);
// p -= lr*direction.
template <Opt O>
__device__ __forceinline__ void sgd1(const SgdConsts& c, float g, float& p, float& buf) {
  if (c.wd_on) g = __fadd_rn(g, __fmul_rn(c.wd, p));
  float d = g;
  if constexpr (O == Opt::SgdMomentum) {
    buf = c.first ? g : __fadd_rn(__fmul_rn(c.mu, buf), __fmul_rn(c.omd, g));
    d = c.nesterov ? __fadd_rn(g, __fmul_rn(c.mu, buf)) : buf;
  }
  p = __fsub_rn(p, __fmul_rn(c.lr, d));
}

// The element update of optimizer O with the (scaled) mean gradient g.
template <Opt O>
__device__ __forceinline__ void update1(const StepArgs& P, float g, float& p, float (&s)[kSA<O>]) {
  if constexpr (O == Opt::AdamW) {
    adam1(P.c, g, p, s[0], s[1]);
  } else {
    sgd1<O>(P.sgd, g, p, s[0]);
  }
}

// Four consecutive elements: rank sums g, parameters p, state streams st.
// Written out per component (no indexed access into the vectors).
template <int NR, Opt O>
__device__ __forceinline__ void update4(const StepArgs& P, float gm, float4 g, float4& p,
                                        float4 (&st)[kSA<O>]) {
  if constexpr (O == Opt::AdamW) {
    adam1(P.c, scaled_mean<NR>(g.x, P, gm), p.x, st[0].x, st[1].x);
    adam1(P.c, scaled_mean<NR>(g.y, P, gm), p.y, st[0].y, st[1].y);
    adam1(P.c, scaled_mean<NR>(g.z, P, gm), p.z, st[0].z, st[1].z);
    adam1(P.c, scaled_mean<NR>(g.w, P, gm), p.w, st[0].w, st[1].w);
  } else {
    sgd1<O>(P.sgd, scaled_mean<NR>(g.x, P, gm), p.x, st[0].x);
    sgd1<O>(P.sgd, scaled_mean<NR>(g.y, P, gm), p.y, st[0].y);
    sgd1<O>(P.sgd, scaled_mean<NR>(g.z, P, gm), p.z, st[0].z);
    sgd1<O>(P.sgd, scaled_mean<NR>(g.w, P, gm), p.w, st[0].w);
  }
}

// ------------------------------------------------------- scalar element path --

template <int NR, bool MIXED, Opt O>
__device__ __forceinline__ void step_scalar(const StepArgs& P, int64_t j, int owner, float gm) {
  const int N = ranks<NR>(P);
  float s, p;
  if constexpr (MIXED) {
    s = bf_one(__ldcs(static_cast<const uint16_t*>(P.grads[0]) + j));
    for (int r = 1; r < N; ++r)
      s = __fadd_rn(s, bf_one(__ldcs(static_cast<const uint16_t*>(P.grads[r]) + j)));
    p = __ldcs(P.master + j);
  } else {
    s = __ldcs(static_cast<const float*>(P.grads[0]) + j);
    for (int r = 1; r < N; ++r) s = __fadd_rn(s, __ldcs(static_cast<const float*>(P.grads[r]) + j));
    p = __ldcs(static_cast<const float*>(P.reps[owner]) + j);
  }
  float st[kSA<O>];
#pragma unroll
  for (int k = 0; k < kStates<O>; ++k) st[k] = __ldcs(state_ptr(P, k) + j);
  update1<O>(P, scaled_mean<NR>(s, P, gm), p, st);
#pragma unroll
  for (int k = 0; k < kStates<O>; ++k) __stcs(state_ptr(P, k) + j, st[k]);
  // Stage 3 (owner_only) keeps only the owner's replica current.
  const int r_lo = P.owner_only ? owner : 0, r_hi = P.owner_only ? owner : N - 1;
  if constexpr (MIXED) {
    __stcs(P.master + j, p);
    const uint16_t h = to_bf(p);
    for (int r = r_lo; r <= r_hi; ++r) __stcs(static_cast<uint16_t*>(P.reps[r]) + j, h);
  } else {
    for (int r = r_lo; r <= r_hi; ++r) __stcs(static_cast<float*>(P.reps[r]) + j, p);
  }
}

// ------------------------------------------------------- fp32 vector path (V=4)

template <int NR, Opt O>
__device__ __forceinline__ void step_vec_fp32(const StepArgs& P, int64_t j, int owner, float gm) {
  const int N = ranks<NR>(P);
  // Loads first: parameter, state, then every rank's gradient.
  float4 p;
  if (j + 3 < P.bounds[owner + 1]) {
    p = ld4(static_cast<const float*>(P.reps[owner]) + j);
  } else {  // the unit straddles a shard boundary: per-element owners
    float e[4];
    int o = owner;
    for (int k = 0; k < 4; ++k) {
      o = advance_owner(P, o, j + k);
      e[k] = __ldcs(static_cast<const float*>(P.reps[o]) + j + k);
    }
    p = make_float4(e[0], e[1], e[2], e[3]);
  }
  float4 st[kSA<O>];
#pragma unroll
  for (int k = 0; k < kStates<O>; ++k) st[k] = ld4(state_ptr(P, k) + j);
  float4 s;
  if constexpr (NR > 0) {
    float4 g[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) g[r] = ld4(static_cast<const float*>(P.grads[r]) + j);
    s = g[0];
#pragma unroll
    for (int r = 1; r < NR; ++r) {
      s.x = __fadd_rn(s.x, g[r].x); s.y = __fadd_rn(s.y, g[r].y);
      s.z = __fadd_rn(s.z, g[r].z); s.w = __fadd_rn(s.w, g[r].w);
    }
  } else {
    s = ld4(static_cast<const float*>(P.grads[0]) + j);
#pragma unroll 4
    for (int r = 1; r < N; ++r) {
      const float4 g = ld4(static_cast<const float*>(P.grads[r]) + j);
      s.x = __fadd_rn(s.x, g.x); s.y = __fadd_rn(s.y, g.y);
      s.z = __fadd_rn(s.z, g.z); s.w = __fadd_rn(s.w, g.w);
    }
  }
  update4<NR, O>(P, gm, s, p, st);
#pragma unroll
  for (int k = 0; k < kStates<O>; ++k) st4(state_ptr(P, k) + j, st[k]);
  if (P.owner_only) {  // stage 3: the owners of the unit's elements only
    const int last = advance_owner(P, owner, j + 3);
    if (last == owner) {
      st4(static_cast<float*>(P.reps[owner]) + j, p);
    } else {
      const float e[4] = {p.x, p.y, p.z, p.w};
      int o = owner;
      for (int k = 0; k < 4; ++k) {
        o = advance_owner(P, o, j + k);
        __stcs(static_cast<float*>(P.reps[o]) + j + k, e[k]);
      }
    }
  } else if constexpr (NR > 0) {
#pragma unroll
    for (int r = 0; r < NR; ++r) st4(static_cast<float*>(P.reps[r]) + j, p);
  } else {
    for (int r = 0; r < N; ++r) st4(static_cast<float*>(P.reps[r]) + j, p);
  }
}

// Units per thread: two for SGD in fp32 with one rank (three loads of a unit
// are too few bytes in flight per thread), one everywhere else. AdamW with one
// rank stays at one: two units take 69 registers (3 blocks per SM) and measured
// 19 % slower, where SGD measured 12 % faster (fp32_25m, N = 1).
template <int NR, bool MIXED, Opt O>
constexpr int kUnits = !MIXED && NR == 1 && O != Opt::AdamW ? 2 : 1;

// Two units of an fp32 step with one rank (kUnits): the second blockDim.x
// units after the first (each warp-wide access still covers 512 contiguous
// bytes), the loads of both issued before any arithmetic. One rank owns every
// index, so no unit straddles a shard. u0 < nvec; the second unit exists when
// u1 < nvec.
template <Opt O>
__device__ __forceinline__ void step_vec_fp32_one_rank(const StepArgs& P, int64_t base,
                                                       int64_t u0, int64_t nvec, float gm) {
  const int64_t u1 = u0 + blockDim.x;
  const bool two = u1 < nvec;
  const int64_t j[2] = {base + u0 * 4, base + u1 * 4};
  const float* rep = static_cast<const float*>(P.reps[0]);
  const float* grad = static_cast<const float*>(P.grads[0]);
  float4 p[2], g[2], st[2][kSA<O>];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    if (u == 1 && !two) break;
    p[u] = ld4(rep + j[u]);
#pragma unroll
    for (int k = 0; k < kStates<O>; ++k) st[u][k] = ld4(state_ptr(P, k) + j[u]);
    g[u] = ld4(grad + j[u]);
  }
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    if (u == 1 && !two) break;
    update4<1, O>(P, gm, g[u], p[u], st[u]);
#pragma unroll
    for (int k = 0; k < kStates<O>; ++k) st4(state_ptr(P, k) + j[u], st[u][k]);
    st4(static_cast<float*>(P.reps[0]) + j[u], p[u]);
  }
}

// ------------------------------------------------------ mixed vector path (V=8)

template <int NR, Opt O>
__device__ __forceinline__ void step_vec_mixed(const StepArgs& P, int64_t j, int owner, float gm) {
  const int N = ranks<NR>(P);
  float4 p4[2] = {ld4(P.master + j), ld4(P.master + j + 4)};
  float4 st[2][kSA<O>];
#pragma unroll
  for (int k = 0; k < kStates<O>; ++k) {
    st[0][k] = ld4(state_ptr(P, k) + j);
    st[1][k] = ld4(state_ptr(P, k) + j + 4);
  }
  float s[8];
  if constexpr (NR > 0) {
    uint4 w[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) w[r] = ld8h(static_cast<const uint16_t*>(P.grads[r]) + j);
    unpack8(w[0], s);
#pragma unroll
    for (int r = 1; r < NR; ++r) {
      float f[8];
      unpack8(w[r], f);
#pragma unroll
      for (int k = 0; k < 8; ++k) s[k] = __fadd_rn(s[k], f[k]);
    }
  } else {
    unpack8(ld8h(static_cast<const uint16_t*>(P.grads[0]) + j), s);
#pragma unroll 4
    for (int r = 1; r < N; ++r) {
      float f[8];
      unpack8(ld8h(static_cast<const uint16_t*>(P.grads[r]) + j), f);
#pragma unroll
      for (int k = 0; k < 8; ++k) s[k] = __fadd_rn(s[k], f[k]);
    }
  }
  update4<NR, O>(P, gm, make_float4(s[0], s[1], s[2], s[3]), p4[0], st[0]);
  update4<NR, O>(P, gm, make_float4(s[4], s[5], s[6], s[7]), p4[1], st[1]);
  st4(P.master + j, p4[0]);
  st4(P.master + j + 4, p4[1]);
#pragma unroll
  for (int k = 0; k < kStates<O>; ++k) {
    st4(state_ptr(P, k) + j, st[0][k]);
    st4(state_ptr(P, k) + j + 4, st[1][k]);
  }
  const float p[8] = {p4[0].x, p4[0].y, p4[0].z, p4[0].w, p4[1].x, p4[1].y, p4[1].z, p4[1].w};
  const uint4 h = pack8(p);
  if (P.owner_only) {  // stage 3: the owners of the unit's elements only
    const int last = advance_owner(P, owner, j + 7);
    if (last == owner) {
      st8h(static_cast<uint16_t*>(P.reps[owner]) + j, h);
    } else {
      int o = owner;
      for (int k = 0; k < 8; ++k) {
        o = advance_owner(P, o, j + k);
        __stcs(static_cast<uint16_t*>(P.reps[o]) + j + k, to_bf(p[k]));
      }
    }
  } else if constexpr (NR > 0) {
#pragma unroll
    for (int r = 0; r < NR; ++r) st8h(static_cast<uint16_t*>(P.reps[r]) + j, h);
  } else {
    for (int r = 0; r < N; ++r) st8h(static_cast<uint16_t*>(P.reps[r]) + j, h);
  }
}

// ------------------------------------------------------------------ kernels --

template <int NR, bool MIXED, Opt O>
__global__ void __launch_bounds__(kThreads) zero_step_kernel(const __grid_constant__ StepArgs P) {
  constexpr int V = MIXED ? 8 : 4;
  const int64_t tid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  const Split& sp = P.sp;
  // A later bucket of the same step (disjoint indices) may start now; this
  // kernel still completes only after the one before it (the wait at the end).
  pdl_allow_next();
  // The squared norm (or the multiplier formed from it) may come from the
  // kernel just before this one (a clipped step chained to its norm): wait
  // for it before reading.
  if (P.norm_sq) pdl_wait_previous();
  const float gm = block_grad_multiplier(P);

  // Scalar head and tail (a handful of elements, or the whole range when the
  // buffers do not share a 16-byte phase). j grows with s, so the owner scan
  // only moves forward.
  const int64_t nscalar = sp.head + sp.tail;
  if (tid < nscalar) {
    const int64_t body_end = sp.lo + sp.head + sp.nvec * V;
    int owner = 0;
    for (int64_t s = tid; s < nscalar; s += stride) {
      const int64_t j = s < sp.head ? sp.lo + s : body_end + (s - sp.head);
      owner = advance_owner(P, owner, j);
      step_scalar<NR, MIXED, O>(P, j, owner, gm);
    }
  }

  // Vector body: one unit per thread, or two (kUnits).
  const int64_t base = sp.lo + sp.head;
  if constexpr (kUnits<NR, MIXED, O> == 2) {
    const int64_t span = 2 * int64_t(blockDim.x);  // units per block and iteration
    for (int64_t b0 = int64_t(blockIdx.x) * span; b0 < sp.nvec; b0 += int64_t(gridDim.x) * span)
      if (b0 + threadIdx.x < sp.nvec)
        step_vec_fp32_one_rank<O>(P, base, b0 + threadIdx.x, sp.nvec, gm);
  } else {
    int owner = 0;
    for (int64_t u = tid; u < sp.nvec; u += stride) {
      const int64_t j = base + u * V;
      if constexpr (MIXED) {
        if (P.owner_only) owner = advance_owner(P, owner, j);
        step_vec_mixed<NR, O>(P, j, owner, gm);
      } else {
        owner = advance_owner(P, owner, j);
        step_vec_fp32<NR, O>(P, j, owner, gm);
      }
    }
  }
  pdl_wait_previous();
}

// ------------------------------------------------- squared global gradient norm

// Deterministic block sum of one double per thread (fixed shuffle tree, then
// warps in order); the result is valid in thread 0.
__device__ __forceinline__ double block_sum(double x) {
  __shared__ double warp_sums[32];
  for (int off = 16; off > 0; off >>= 1) x += __shfl_down_sync(0xffffffffu, x, off);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) warp_sums[warp] = x;
  __syncthreads();
  double t = 0.0;
  if (threadIdx.x == 0) {
    for (int w = 0; w < int(blockDim.x >> 5); ++w) t += warp_sums[w];
  }
  __syncthreads();
  return t;
}

// Running sum of squares of floats, accurate to about double precision while
// spending float operations only (the GPU's double rate is low): every square
// is split exactly into p + e with p = fl(x*x), e = fma(x, x, -p); the p are
// added with Neumaier's compensated summation (s, c) and the small e directly.
// Squares outside the normal float range (|x| > 2^60, or 0 < |x| < 2^-60) go
// to a double accumulator instead. value() adds the parts in double.
// The rare out-of-range square, kept out of line so the common path carries no
// double-precision instruction (a branch, not a predicated sequence).
__device__ __noinline__ double add_wide_square(double wide, float x) {
  return wide + double(x) * double(x);
}

struct SquareSum {
  float s = 0.0f, c = 0.0f, e = 0.0f;
  double wide = 0.0;
  __device__ __forceinline__ void add(float x) {
    const float ax = fabsf(x);
    if (ax > 0x1p60f || (ax < 0x1p-60f && ax != 0.0f)) {
      wide = add_wide_square(wide, x);
      return;
    }
    const float p = __fmul_rn(x, x);
    e = __fadd_rn(e, fmaf(x, x, -p));
    const float t = __fadd_rn(s, p);
    c = __fadd_rn(c, s >= p ? __fadd_rn(__fsub_rn(s, t), p) : __fadd_rn(__fsub_rn(p, t), s));
    s = t;
  }
  __device__ __forceinline__ double value() const {
    return (double(s) + double(c)) + (double(e) + wide);
  }
};

// Partial sums of ||mean gradient||^2. Partial c < nchunks covers the vector
// units [c*U, (c+1)*U) with U = P.chunk / V; partial nchunks covers the
// scalar head and tail. Every thread accumulates the squares of the float
// means of its elements (SquareSum), then blocks reduce in double in a fixed
// order, so every partial -- and the total -- is independent of the grid size.
template <int NR, bool BF16>
__device__ __forceinline__ double norm_chunk_sum(const NormArgs& P, int64_t c) {
  constexpr int V = BF16 ? 8 : 4;
  const int64_t U = P.chunk / V;
  const int N = NR > 0 ? NR : P.N;
  const Split& sp = P.sp;
  const int64_t base = sp.lo + sp.head;
  SquareSum acc;
  if (c < P.nchunks) {
    const int64_t u_end = (c + 1) * U < sp.nvec ? (c + 1) * U : sp.nvec;
    // Two units per thread per iteration: every load of both is issued before
    // any arithmetic. The element order within the thread is fixed, so the
    // partial stays independent of the grid.
    for (int64_t u0 = c * U + threadIdx.x; u0 < u_end; u0 += 2 * blockDim.x) {
      const int64_t u1 = u0 + blockDim.x;
      const bool has1 = u1 < u_end;
      const int64_t j0 = base + u0 * V, j1 = base + (has1 ? u1 : u0) * V;
      float s0[V], s1[V];
      if constexpr (BF16) {
        unpack8(ld8h(static_cast<const uint16_t*>(P.grads[0]) + j0), s0);
        unpack8(ld8h(static_cast<const uint16_t*>(P.grads[0]) + j1), s1);
        for (int r = 1; r < N; ++r) {
          float f0[8], f1[8];
          unpack8(ld8h(static_cast<const uint16_t*>(P.grads[r]) + j0), f0);
          unpack8(ld8h(static_cast<const uint16_t*>(P.grads[r]) + j1), f1);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            s0[k] = __fadd_rn(s0[k], f0[k]);
            s1[k] = __fadd_rn(s1[k], f1[k]);
          }
        }
      } else {
        float4 a = ld4(static_cast<const float*>(P.grads[0]) + j0);
        float4 b = ld4(static_cast<const float*>(P.grads[0]) + j1);
        for (int r = 1; r < N; ++r) {
          const float4 x = ld4(static_cast<const float*>(P.grads[r]) + j0);
          const float4 y = ld4(static_cast<const float*>(P.grads[r]) + j1);
          a.x = __fadd_rn(a.x, x.x); a.y = __fadd_rn(a.y, x.y);
          a.z = __fadd_rn(a.z, x.z); a.w = __fadd_rn(a.w, x.w);
          b.x = __fadd_rn(b.x, y.x); b.y = __fadd_rn(b.y, y.y);
          b.z = __fadd_rn(b.z, y.z); b.w = __fadd_rn(b.w, y.w);
        }
        s0[0] = a.x; s0[1] = a.y; s0[2] = a.z; s0[3] = a.w;
        s1[0] = b.x; s1[1] = b.y; s1[2] = b.z; s1[3] = b.w;
      }
#pragma unroll
      for (int k = 0; k < V; ++k) acc.add(mean_of<NR>(s0[k], P.fN));
      if (has1) {
#pragma unroll
        for (int k = 0; k < V; ++k) acc.add(mean_of<NR>(s1[k], P.fN));
      }
    }
  } else {
    const int64_t nscalar = sp.head + sp.tail;
    const int64_t body_end = base + sp.nvec * V;
    for (int64_t t = threadIdx.x; t < nscalar; t += blockDim.x) {
      const int64_t j = t < sp.head ? sp.lo + t : body_end + (t - sp.head);
      float s;
      if constexpr (BF16) {
        s = bf_one(__ldcs(static_cast<const uint16_t*>(P.grads[0]) + j));
        for (int r = 1; r < N; ++r)
          s = __fadd_rn(s, bf_one(__ldcs(static_cast<const uint16_t*>(P.grads[r]) + j)));
      } else {
        s = __ldcs(static_cast<const float*>(P.grads[0]) + j);
        for (int r = 1; r < N; ++r)
          s = __fadd_rn(s, __ldcs(static_cast<const float*>(P.grads[r]) + j));
      }
      acc.add(mean_of<NR>(s, P.fN));
    }
  }
  return block_sum(acc.value());
}

template <int NR, bool BF16>
__global__ void __launch_bounds__(kThreads)
    grad_norm_partials_kernel(const __grid_constant__ NormArgs P) {
  // a step that forms the total itself may start now: it waits for this
  // kernel to complete before it reads a partial
  pdl_allow_next();
  for (int64_t c = P.c_begin + blockIdx.x; c < P.c_end; c += gridDim.x) {
    const double total = norm_chunk_sum<NR, BF16>(P, c);
    if (threadIdx.x == 0) P.partials[c] = total;
  }
}

// The partials added in a fixed order by one block (fixed_order_total). It is
// launched as a programmatic dependent of the partials: it lets the step after
// it start, then waits for the partials before it reads them.
__global__ void __launch_bounds__(kThreads) grad_norm_total_kernel(const __grid_constant__ NormArgs P) {
  pdl_allow_next();
  pdl_wait_previous();
  const double total = fixed_order_total(P.partials, P.nchunks + 1);
  if (threadIdx.x == 0) {
    *P.out = total;
    if (P.gm_out) *P.gm_out = clip_multiplier(P.gscale, P.max_norm, total);
  }
}

// One element of the DDP mean, in place in every rank's buffer.
template <int NR, bool BF16>
__device__ __forceinline__ void mean_scalar(const AllreduceArgs& P, int64_t j) {
  const int N = NR > 0 ? NR : P.N;
  if constexpr (BF16) {
    float acc = bf_one(__ldcs(static_cast<const uint16_t*>(P.grads[0]) + j));
    for (int r = 1; r < N; ++r)
      acc = __fadd_rn(acc, bf_one(__ldcs(static_cast<const uint16_t*>(P.grads[r]) + j)));
    const uint16_t h = to_bf(mean_of<NR>(acc, P.fN));
    for (int r = 0; r < N; ++r) __stcs(static_cast<uint16_t*>(P.grads[r]) + j, h);
  } else {
    float acc = __ldcs(static_cast<const float*>(P.grads[0]) + j);
    for (int r = 1; r < N; ++r)
      acc = __fadd_rn(acc, __ldcs(static_cast<const float*>(P.grads[r]) + j));
    const float g = mean_of<NR>(acc, P.fN);
    for (int r = 0; r < N; ++r) __stcs(static_cast<float*>(P.grads[r]) + j, g);
  }
}

template <int NR, bool BF16>
__global__ void __launch_bounds__(kThreads)
    allreduce_mean_kernel(const __grid_constant__ AllreduceArgs P) {
  constexpr int V = BF16 ? 8 : 4;
  const int N = NR > 0 ? NR : P.N;
  const int64_t tid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  const Split& sp = P.sp;

  const int64_t nscalar = sp.head + sp.tail;
  const int64_t body_end = sp.lo + sp.head + sp.nvec * V;
  for (int64_t s = tid; s < nscalar; s += stride) {
    const int64_t j = s < sp.head ? sp.lo + s : body_end + (s - sp.head);
    mean_scalar<NR, BF16>(P, j);
  }

  const int64_t base = sp.lo + sp.head;
  for (int64_t u = tid; u < sp.nvec; u += stride) {
    const int64_t j = base + u * V;
    if constexpr (BF16) {
      float s[8];
      unpack8(ld8h(static_cast<const uint16_t*>(P.grads[0]) + j), s);
#pragma unroll 4
      for (int r = 1; r < N; ++r) {
        float f[8];
        unpack8(ld8h(static_cast<const uint16_t*>(P.grads[r]) + j), f);
#pragma unroll
        for (int k = 0; k < 8; ++k) s[k] = __fadd_rn(s[k], f[k]);
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) s[k] = mean_of<NR>(s[k], P.fN);
      const uint4 h = pack8(s);
      for (int r = 0; r < N; ++r) st8h(static_cast<uint16_t*>(P.grads[r]) + j, h);
    } else {
      float4 s = ld4(static_cast<const float*>(P.grads[0]) + j);
#pragma unroll 4
      for (int r = 1; r < N; ++r) {
        const float4 g = ld4(static_cast<const float*>(P.grads[r]) + j);
        s.x = __fadd_rn(s.x, g.x); s.y = __fadd_rn(s.y, g.y);
        s.z = __fadd_rn(s.z, g.z); s.w = __fadd_rn(s.w, g.w);
      }
      s.x = mean_of<NR>(s.x, P.fN); s.y = mean_of<NR>(s.y, P.fN);
      s.z = mean_of<NR>(s.z, P.fN); s.w = mean_of<NR>(s.w, P.fN);
      for (int r = 0; r < N; ++r) st4(static_cast<float*>(P.grads[r]) + j, s);
    }
  }
}

// ------------------------------------------------------- stage-3 all-gather --

// Every replica receives each shard from its owner's replica: one 16-byte load
// and N-1 16-byte stores per unit (V = 4 fp32 or 8 bf16 elements); a unit that
// straddles a shard boundary, and the scalar head and tail, go element by
// element. A pure copy: the bits are moved, never converted.
__device__ __forceinline__ int gather_owner(const GatherArgs& P, int owner, int64_t j) {
  while (j >= P.bounds[owner + 1]) ++owner;
  return owner;
}

template <typename E>
__device__ __forceinline__ void gather_one(const GatherArgs& P, int owner, int64_t j) {
  const E x = __ldcs(static_cast<const E*>(P.reps[owner]) + j);
  for (int r = 0; r < P.N; ++r)
    if (r != owner) __stcs(static_cast<E*>(P.reps[r]) + j, x);
}

// U units per thread per iteration, block-interleaved (unit u of a thread is
// u * blockDim.x units after its first, so each warp-wide access covers 512
// contiguous bytes): the loads of all U units, each from its unit's owner, are
// issued before any store, then each unit goes to the N-1 other replicas. The
// owner scan only moves forward along a thread's units.
template <bool BF16, int U>
__global__ void __launch_bounds__(kThreads) gather_kernel(const __grid_constant__ GatherArgs P) {
  using E = typename std::conditional<BF16, uint16_t, float>::type;
  constexpr int V = 16 / int(sizeof(E));
  const int64_t tid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  const Split& sp = P.sp;

  const int64_t nscalar = sp.head + sp.tail;
  const int64_t body_end = sp.lo + sp.head + sp.nvec * V;
  int owner = 0;
  for (int64_t s = tid; s < nscalar; s += stride) {
    const int64_t j = s < sp.head ? sp.lo + s : body_end + (s - sp.head);
    owner = gather_owner(P, owner, j);
    gather_one<E>(P, owner, j);
  }

  const int64_t base = sp.lo + sp.head;
  const int64_t span = int64_t(blockDim.x) * U;  // units per block and iteration
  owner = 0;
  for (int64_t b0 = int64_t(blockIdx.x) * span; b0 < sp.nvec; b0 += int64_t(gridDim.x) * span) {
    uint4 x[U];
    int o[U];
    bool whole[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t uv = b0 + threadIdx.x + int64_t(u) * blockDim.x;
      whole[u] = false;
      o[u] = owner;
      if (uv < sp.nvec) {
        const int64_t j = base + uv * V;
        owner = gather_owner(P, owner, j);
        o[u] = owner;
        whole[u] = j + V - 1 < P.bounds[owner + 1];
        if (whole[u])
          x[u] = __ldcs(reinterpret_cast<const uint4*>(static_cast<const E*>(P.reps[owner]) + j));
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t uv = b0 + threadIdx.x + int64_t(u) * blockDim.x;
      if (uv >= sp.nvec) continue;
      const int64_t j = base + uv * V;
      if (whole[u]) {
        for (int r = 0; r < P.N; ++r)
          if (r != o[u]) __stcs(reinterpret_cast<uint4*>(static_cast<E*>(P.reps[r]) + j), x[u]);
      } else {  // the unit straddles a shard boundary: element by element
        int e = o[u];
        for (int k = 0; k < V; ++k) {
          e = gather_owner(P, e, j + k);
          gather_one<E>(P, e, j + k);
        }
      }
    }
  }
}

// m = v = 0 (each when present) and (mixed) master = init over the split range.
__global__ void __launch_bounds__(kThreads) init_state_kernel(const __grid_constant__ InitArgs P) {
  const int64_t tid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  const Split& sp = P.sp;
  const int64_t nscalar = sp.head + sp.tail;
  const int64_t body_end = sp.lo + sp.head + sp.nvec * 4;
  for (int64_t s = tid; s < nscalar; s += stride) {
    const int64_t j = s < sp.head ? sp.lo + s : body_end + (s - sp.head);
    if (P.m) P.m[j] = 0.0f;
    if (P.v) P.v[j] = 0.0f;
    if (P.master) P.master[j] = P.init[j];
  }
  const int64_t base = sp.lo + sp.head;
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int64_t u = tid; u < sp.nvec; u += stride) {
    const int64_t j = base + u * 4;
    if (P.m) st4(P.m + j, z);
    if (P.v) st4(P.v + j, z);
    if (P.master) st4(P.master + j, ld4(P.init + j));
  }
}

}  // namespace
}  // namespace zk

namespace zk {
namespace {

// ------------------------------------------------------------ grid sizing --

int sm_count() {
  static int cached[256] = {0};  // indexed by device ordinal
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev < 0 || dev >= int(sizeof(cached) / sizeof(cached[0]))) return 0;
  if (cached[dev] == 0) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev] = sms;
  }
  return cached[dev];
}

// Blocks for `work` thread-iterations: enough to cover it, at most the number
// of blocks resident at once on the whole GPU (a persistent-style grid).
template <typename K>
cudaError_t grid_for(K kernel, int64_t work, int* blocks) {
  int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, 0);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const int64_t cap = int64_t(sms) * per_sm;
  int64_t need = (work + kThreads - 1) / kThreads;
  if (need < 1) need = 1;
  *blocks = int(need < cap ? need : cap);
  return cudaSuccess;
}

template <typename K, typename A>
cudaError_t launch(K kernel, const A& args, int64_t work, cudaStream_t s) {
  int blocks = 0;
  cudaError_t e = grid_for(kernel, work, &blocks);
  if (e != cudaSuccess) return e;
  kernel<<<blocks, kThreads, 0, s>>>(args);
  return cudaGetLastError();
}

// One pass: blocks for all the work, launched in waves, each block taking
// one stretch of units and exiting (no grid-stride loop). For the gather
// (1 read, N-1 writes) this measured 6-13 % faster than a persistent
// grid-stride grid of the same kernel, and than the bulk-copy pipeline it
// replaced, at N = 2, 4, 8 on 25M-320M elements.
template <typename K, typename A>
cudaError_t launch_one_pass(K kernel, const A& args, int64_t threads_needed, cudaStream_t s,
                            bool dependent = false) {
  int64_t blocks = (threads_needed + kThreads - 1) / kThreads;
  if (blocks < 1) blocks = 1;
  if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
  if (!dependent) {
    kernel<<<unsigned(blocks), kThreads, 0, s>>>(args);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(blocks));
  cfg.blockDim = dim3(unsigned(kThreads));
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args);
}

// The step: register streaming in one pass, as a programmatic dependent of the
// kernel before it when the caller asks (a later bucket of one step, or a
// clipped step after its norm). fp32 AdamW with one rank and no such chain
// keeps a persistent grid-stride grid, measured 2 % faster there; SGD with
// one rank takes two units per thread (kUnits).
template <bool MIXED, Opt O>
cudaError_t launch_step_t(const StepArgs& a, cudaStream_t s) {
  const int64_t nscalar = a.sp.head + a.sp.tail;
  const bool two = a.N == 1 && kUnits<1, MIXED, O> == 2;
  const int64_t body = two ? (a.sp.nvec + 1) / 2 : a.sp.nvec;
  const int64_t work = body > nscalar ? body : nscalar;
  const bool dep = a.dependent != 0;
  if (a.sp.nvec == 0 || (!MIXED && O == Opt::AdamW && a.N == 1 && !dep)) {
    switch (a.N) {
      case 1: return launch(zero_step_kernel<1, MIXED, O>, a, work, s);
      case 2: return launch(zero_step_kernel<2, MIXED, O>, a, work, s);
      case 4: return launch(zero_step_kernel<4, MIXED, O>, a, work, s);
      case 8: return launch(zero_step_kernel<8, MIXED, O>, a, work, s);
      default: return launch(zero_step_kernel<0, MIXED, O>, a, work, s);
    }
  }
  switch (a.N) {
    case 1: return launch_one_pass(zero_step_kernel<1, MIXED, O>, a, work, s, dep);
    case 2: return launch_one_pass(zero_step_kernel<2, MIXED, O>, a, work, s, dep);
    case 4: return launch_one_pass(zero_step_kernel<4, MIXED, O>, a, work, s, dep);
    case 8: return launch_one_pass(zero_step_kernel<8, MIXED, O>, a, work, s, dep);
    default: return launch_one_pass(zero_step_kernel<0, MIXED, O>, a, work, s, dep);
  }
}

template <Opt O>
cudaError_t launch_step_o(const StepArgs& a, bool mixed, cudaStream_t s) {
  return mixed ? launch_step_t<true, O>(a, s) : launch_step_t<false, O>(a, s);
}

// The DDP mean: register streaming in one pass over a vector body (5-6 %
// faster than the bulk-copy pipeline it replaced on fp32_25m, gpt2_small and
// fp32_320m), the grid-stride grid for a scalar-only range.
template <bool BF16>
cudaError_t launch_allreduce_t(const AllreduceArgs& a, cudaStream_t s) {
  const int64_t work = a.sp.nvec > a.sp.head + a.sp.tail ? a.sp.nvec : a.sp.head + a.sp.tail;
  if (a.sp.nvec > 0) {
    switch (a.N) {
      case 1: return launch_one_pass(allreduce_mean_kernel<1, BF16>, a, work, s);
      case 2: return launch_one_pass(allreduce_mean_kernel<2, BF16>, a, work, s);
      case 4: return launch_one_pass(allreduce_mean_kernel<4, BF16>, a, work, s);
      case 8: return launch_one_pass(allreduce_mean_kernel<8, BF16>, a, work, s);
      default: return launch_one_pass(allreduce_mean_kernel<0, BF16>, a, work, s);
    }
  }
  switch (a.N) {
    case 1: return launch(allreduce_mean_kernel<1, BF16>, a, work, s);
    case 2: return launch(allreduce_mean_kernel<2, BF16>, a, work, s);
    case 4: return launch(allreduce_mean_kernel<4, BF16>, a, work, s);
    case 8: return launch(allreduce_mean_kernel<8, BF16>, a, work, s);
    default: return launch(allreduce_mean_kernel<0, BF16>, a, work, s);
  }
}

}  // namespace

cudaError_t launch_step(const StepArgs& a, bool mixed, Opt opt, cudaStream_t s) {
  switch (opt) {
    case Opt::AdamW: return launch_step_o<Opt::AdamW>(a, mixed, s);
    case Opt::SgdMomentum: return launch_step_o<Opt::SgdMomentum>(a, mixed, s);
    case Opt::Sgd: return launch_step_o<Opt::Sgd>(a, mixed, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_allreduce(const AllreduceArgs& a, bool bf16, cudaStream_t s) {
  return bf16 ? launch_allreduce_t<true>(a, s) : launch_allreduce_t<false>(a, s);
}

cudaError_t launch_init(const InitArgs& a, cudaStream_t s) {
  const int64_t work = a.sp.nvec > a.sp.head + a.sp.tail ? a.sp.nvec : a.sp.head + a.sp.tail;
  return launch(init_state_kernel, a, work, s);
}

namespace {
template <bool BF16>
cudaError_t launch_gather_t(const GatherArgs& a, cudaStream_t s) {
  // Units per thread: one with at least four replicas, two below (fewer
  // stores per load); measured at N = 2, 4, 8 (6.1, 6.5, 6.7 TB/s).
  const int64_t nscalar = a.sp.head + a.sp.tail;
  if (a.N >= 4) {
    const int64_t work = a.sp.nvec > nscalar ? a.sp.nvec : nscalar;
    return launch_one_pass(gather_kernel<BF16, 1>, a, work, s);
  }
  const int64_t units = (a.sp.nvec + 1) / 2;
  return launch_one_pass(gather_kernel<BF16, 2>, a, units > nscalar ? units : nscalar, s);
}
}  // namespace

cudaError_t launch_gather(const GatherArgs& a, bool bf16, cudaStream_t s) {
  return bf16 ? launch_gather_t<true>(a, s) : launch_gather_t<false>(a, s);
}

namespace {
template <bool BF16>
cudaError_t launch_partials_t(const NormArgs& a, cudaStream_t s) {
  if (a.c_end <= a.c_begin) return cudaSuccess;
  const int64_t work = (a.c_end - a.c_begin) * kThreads;  // one block per partial at most
  switch (a.N) {
    case 1: return launch(grad_norm_partials_kernel<1, BF16>, a, work, s);
    case 2: return launch(grad_norm_partials_kernel<2, BF16>, a, work, s);
    case 4: return launch(grad_norm_partials_kernel<4, BF16>, a, work, s);
    case 8: return launch(grad_norm_partials_kernel<8, BF16>, a, work, s);
    default: return launch(grad_norm_partials_kernel<0, BF16>, a, work, s);
  }
}
}  // namespace

cudaError_t launch_norm_partials(const NormArgs& a, bool bf16, cudaStream_t s) {
  return bf16 ? launch_partials_t<true>(a, s) : launch_partials_t<false>(a, s);
}

cudaError_t launch_norm_total(const NormArgs& a, cudaStream_t s) {
  return launch_one_pass(grad_norm_total_kernel, a, kThreads, s, true);
}

cudaError_t launch_norm(const NormArgs& a, bool bf16, cudaStream_t s) {
  NormArgs all = a;
  all.c_begin = 0;
  all.c_end = a.nchunks + 1;
  cudaError_t e = launch_norm_partials(all, bf16, s);
  if (e != cudaSuccess) return e;
  return launch_norm_total(all, s);
}

// ---------------------------------------------- partial sums without allocation
//
// Scratch for zero_grad_norm_sq_noalloc: the partial sums live in this fixed
// array, which every GPU that loads the library keeps (512 KB) until the
// process exits. Every call shares it and leaves its partials behind; each
// partial a call reads was written earlier in that same call, so nothing has
// to start at zero. Calls whose work overlaps on the GPU race on it.
static __device__ __align__(256) double g_noalloc_partials[kNoAllocPartials];

cudaError_t noalloc_partials(double** ptr) {
  // In host code g_noalloc_partials is only a stand-in for the device array;
  // its device address is looked up once per device, with that device current.
  static std::mutex mu;
  static double* addr[256] = {nullptr};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 256) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_partials);
    if (e != cudaSuccess) return e;
    addr[dev] = static_cast<double*>(p);
  }
  *ptr = addr[dev];
  return cudaSuccess;
}

}  // namespace zk
