// Host side of libzero_gb300.so: argument checking, the shard planner, memory
// accounting, per-step constants, the bucket streamer, and error reporting.
// Device work is delegated to the launchers in zero_kernels.cu.
//
// Built with -ffp-contract=off so that the per-step constants are formed with
// separately rounded double operations.

#include <algorithm>
#include <chrono>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <thread>
#include <vector>

#include "zero_internal.h"

struct zero_states {
  int64_t n;
  int32_t N;
  int32_t precision;
  float* m;
  float* v;
  float* master;
  int64_t bounds[ZERO_MAX_RANKS + 1];
  // Events of the host-input pipeline (created on first use, reused by later
  // calls, destroyed with the handle).
  std::vector<cudaEvent_t> events;
  // Step launches on this handle so far, and the chunking of the last
  // host-input call with the launch count right after it: when nothing else
  // was launched since, the next host-input call with the same chunking and
  // staging buffers may start copying a chunk as soon as the previous call's
  // step on that chunk is done.
  uint64_t launches = 0;
  uint64_t host_launches = ~uint64_t(0);
  int64_t host_B = 0;
  std::vector<void*> host_staging;
};

namespace {

thread_local char g_last_error[512] = "";

// Handle allocations of this thread still to fail (zero_debug_fail_host_allocs).
thread_local int32_t g_failing_allocs = 0;

// A handle from the host allocator, or NULL when it fails (or an injected
// failure is pending for this thread).
template <typename T>
T* new_handle() {
  if (g_failing_allocs > 0) {
    --g_failing_allocs;
    return nullptr;
  }
  return new (std::nothrow) T;
}

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(ZERO_ECUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

bool valid_ranks(int32_t N) { return N >= 1 && N <= ZERO_MAX_RANKS; }

// Shard offsets of np.array_split(np.arange(n), N): a_i = i*q + min(i, r).
void shard_bounds(int64_t n, int32_t N, int64_t* b) {
  const int64_t q = n / N, r = n % N;
  for (int32_t i = 0; i <= N; ++i) b[i] = i * q + std::min<int64_t>(i, r);
}

// ----------------------------------------------------------- alignment plan --

// Element phase of a pointer within a 16-byte line, or -1 if it is not aligned
// to its element size.
int phase_of(const void* p, int elem) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  if (a % elem) return -1;
  return int((a / elem) % (16 / elem));
}

zk::Split make_split(int64_t lo, int64_t hi, bool vector_ok, int phase, int V) {
  zk::Split s{lo, hi - lo, 0, 0};
  if (!vector_ok) return s;
  const int64_t len = hi - lo;
  int64_t head = (V - (phase + lo % V) % V) % V;
  if (head > len) head = len;
  s.head = head;
  s.nvec = (len - head) / V;
  s.tail = len - head - s.nvec * V;
  return s;
}

struct Range {
  uintptr_t lo, hi;
  const char* what;
};

// Every buffer must be disjoint from every other one.
int check_disjoint(std::vector<Range>& rs) {
  std::sort(rs.begin(), rs.end(), [](const Range& a, const Range& b) { return a.lo < b.lo; });
  for (size_t i = 1; i < rs.size(); ++i) {
    if (rs[i].lo < rs[i - 1].hi)
      return fail(ZERO_EINVAL, "buffers overlap (%s and %s)", rs[i - 1].what, rs[i].what);
  }
  return ZERO_OK;
}

// ------------------------------------------------------- step preparation --

int adam_consts(int64_t t, double lr, double beta1, double beta2, double eps, double wd,
                zk::AdamConsts* c) {
  if (t < 1) return fail(ZERO_EINVAL, "step number t=%lld must be >= 1", (long long)t);
  if (!(beta1 >= 0.0 && beta1 < 1.0) || !(beta2 >= 0.0 && beta2 < 1.0))
    return fail(ZERO_EINVAL, "betas must lie in [0, 1) (got %g, %g)", beta1, beta2);
  if (!std::isfinite(lr) || lr < 0.0) return fail(ZERO_EINVAL, "lr must be finite and >= 0");
  if (!std::isfinite(eps) || eps < 0.0) return fail(ZERO_EINVAL, "eps must be finite and >= 0");
  if (!std::isfinite(wd)) return fail(ZERO_EINVAL, "weight_decay must be finite");
  const double td = double(t);
  const double bc1 = 1.0 - std::pow(beta1, td);
  const double bc2 = 1.0 - std::pow(beta2, td);
  c->decay = float(1.0 - lr * wd);
  c->b1 = float(beta1);
  c->omb1 = float(1.0 - beta1);
  c->b2 = float(beta2);
  c->omb2 = float(1.0 - beta2);
  c->step = float(lr / bc1);
  c->bc2s = float(std::sqrt(bc2));
  c->eps = float(eps);
  if (!(c->bc2s > 0.0f)) return fail(ZERO_EINVAL, "1 - beta2^t rounds to zero");
  return ZERO_OK;
}

// Checks the buffers of a step with optimizer `opt` and fills everything in
// StepArgs except the split and the constants.
int prepare_step(void* const* params, const void* const* grads, const zero_states* st,
                 zk::Opt opt, zk::StepArgs* a, bool* vector_ok, int* phase,
                 std::vector<Range>* ranges = nullptr) {
  if (!st) return fail(ZERO_EINVAL, "state handle is NULL");
  if (!params || !grads) return fail(ZERO_EINVAL, "params/grads array is NULL");
  const int nstates = opt == zk::Opt::AdamW ? 2 : (opt == zk::Opt::SgdMomentum ? 1 : 0);
  if (st->n > 0 && nstates >= 1 && !st->m)
    return fail(ZERO_EINVAL, "the state has no first buffer (m), which this optimizer needs");
  if (st->n > 0 && nstates >= 2 && !st->v)
    return fail(ZERO_EINVAL, "the state has no second moment (v): initialised for SGD");
  const int32_t N = st->N;
  const bool mixed = st->precision == ZERO_BF16_MIXED;
  const int es = mixed ? 2 : 4;
  std::memset(a, 0, sizeof(*a));
  a->N = N;
  a->fN = float(N);
  a->norm_sq = nullptr;  // no clipping
  a->gscale = 1.0;       // mean gradient used as is
  a->max_norm = 0.0;
  a->m = st->m;
  a->v = st->v;
  a->master = st->master;
  std::memcpy(a->bounds, st->bounds, sizeof(int64_t) * (N + 1));
  std::vector<Range> rs;
  rs.reserve(2 * N + 3);
  const uintptr_t pbytes = uintptr_t(st->n) * es, sbytes = uintptr_t(st->n) * 4;
  int ph16 = -2, ph32 = -2;
  bool same = true;
  auto note = [&](const void* p, int elem, int* ph) {
    const int q = phase_of(p, elem);
    if (q < 0) return false;
    if (*ph == -2) *ph = q;
    else if (*ph != q) same = false;
    return true;
  };
  for (int32_t r = 0; r < N; ++r) {
    if (st->n > 0 && (!params[r] || !grads[r]))
      return fail(ZERO_EINVAL, "params[%d] or grads[%d] is NULL", r, r);
    a->reps[r] = params[r];
    a->grads[r] = grads[r];
    int* ph = mixed ? &ph16 : &ph32;
    if (!note(params[r], es, ph) || !note(grads[r], es, ph))
      return fail(ZERO_EALIGN, "params[%d]/grads[%d] not aligned to %d bytes", r, r, es);
    if (st->n > 0) {
      rs.push_back({uintptr_t(params[r]), uintptr_t(params[r]) + pbytes, "a parameter replica"});
      rs.push_back({uintptr_t(grads[r]), uintptr_t(grads[r]) + pbytes, "a gradient"});
    }
  }
  const float* sbufs[3] = {st->m, st->v, st->master};
  for (int k = 0; k < 3; ++k) {
    const bool used = k < nstates || (k == 2 && mixed);
    if (!used) continue;
    if (!note(sbufs[k], 4, &ph32)) return fail(ZERO_EALIGN, "state buffer not 4-byte aligned");
    if (st->n > 0) rs.push_back({uintptr_t(sbufs[k]), uintptr_t(sbufs[k]) + sbytes, "a state buffer"});
  }
  if (int e = check_disjoint(rs)) return e;
  if (ranges) *ranges = rs;
  if (mixed) {
    // 8-element units: bf16 buffers 16-byte aligned at j = -ph16 (mod 8), fp32
    // buffers at j = -ph32 (mod 4); both hold when ph16 = ph32 (mod 4).
    *vector_ok = same && (ph16 % 4) == ph32;
    *phase = ph16;
  } else {
    *vector_ok = same;
    *phase = ph32;
  }
  return ZERO_OK;
}

int launch_range(zk::StepArgs& a, zero_states* st, bool vector_ok, int phase, int64_t lo,
                 int64_t hi, cudaStream_t s, zk::Opt opt = zk::Opt::AdamW) {
  if (hi <= lo) return ZERO_OK;
  ++st->launches;
  const bool mixed = st->precision == ZERO_BF16_MIXED;
  a.sp = make_split(lo, hi, vector_ok, phase, mixed ? 8 : 4);
  // gscale * 1 rounded to float once, as the device forms it when clipping
  a.gm = float(a.gscale);
  cudaError_t e = zk::launch_step(a, mixed, opt, s);
  if (e != cudaSuccess) return cuda_fail(e, "zero_step kernel launch");
  return ZERO_OK;
}

int bucket_elems(int32_t precision, int64_t bucket_bytes, int64_t* B) {
  int es;
  if (precision == ZERO_FP32) es = 4;
  else if (precision == ZERO_BF16_MIXED) es = 2;
  else return fail(ZERO_EINVAL, "bucket plan needs precision FP32 or BF16_MIXED");
  if (bucket_bytes < es) return fail(ZERO_EINVAL, "bucket of %lld bytes holds no element",
                                     (long long)bucket_bytes);
  *B = bucket_bytes / es;
  return ZERO_OK;
}

int64_t bucket_count_of(int64_t n, int64_t B) { return n == 0 ? 0 : (n + B - 1) / B; }

void bucket_range_of(int64_t n, int64_t B, int64_t k, int64_t* lo, int64_t* hi) {
  *hi = n - k * B;
  *lo = std::max<int64_t>(0, *hi - B);
}

// Checked a*b + c for the memory totals.
bool mul_add(uint64_t a, uint64_t b, uint64_t* acc) {
  if (a != 0 && b > UINT64_MAX / a) return false;
  const uint64_t p = a * b;
  if (*acc > UINT64_MAX - p) return false;
  *acc += p;
  return true;
}

// Checks the gradients of a norm pass and fills NormArgs except the buffers.
int prepare_norm(const void* const* grads, int64_t n, int32_t N, int32_t precision,
                 zk::NormArgs* a) {
  if (n < 0) return fail(ZERO_EINVAL, "n=%lld must be >= 0", (long long)n);
  if (!valid_ranks(N)) return fail(ZERO_EINVAL, "N=%d outside [1, %d]", N, ZERO_MAX_RANKS);
  if (precision != ZERO_FP32 && precision != ZERO_BF16_MIXED)
    return fail(ZERO_EINVAL, "gradient precision must be FP32 or BF16_MIXED");
  if (!grads) return fail(ZERO_EINVAL, "grads array is NULL");
  const int es = precision == ZERO_BF16_MIXED ? 2 : 4;
  const int V = es == 2 ? 8 : 4;
  std::memset(a, 0, sizeof(*a));
  a->N = N;
  a->fN = float(N);
  int ph = -2;
  bool same = true;
  for (int32_t r = 0; r < N; ++r) {
    if (n > 0 && !grads[r]) return fail(ZERO_EINVAL, "grads[%d] is NULL", r);
    const int q = phase_of(grads[r], es);
    if (q < 0) return fail(ZERO_EALIGN, "grads[%d] not aligned to %d bytes", r, es);
    if (ph == -2) ph = q;
    else if (ph != q) same = false;
    a->grads[r] = grads[r];
  }
  a->sp = make_split(0, n, same, ph, V);
  a->chunk = zk::kNormChunk;
  a->nchunks = (a->sp.nvec * V + a->chunk - 1) / a->chunk;
  a->c_begin = 0;
  a->c_end = a->nchunks + 1;
  return ZERO_OK;
}

// A norm pass into caller scratch: after prepare_norm, checks the scratch and
// the output scalar (aligned, large enough, disjoint from each other and from
// `others`, the call's other buffers) and sets them in `a`.
int attach_norm_buffers(double* scratch, int64_t scratch_count, double* norm_sq,
                        std::vector<Range> others, zk::NormArgs* a) {
  if (!scratch || !norm_sq) return fail(ZERO_EINVAL, "norm scratch or norm_sq is NULL");
  if (reinterpret_cast<uintptr_t>(scratch) % 8 || reinterpret_cast<uintptr_t>(norm_sq) % 8)
    return fail(ZERO_EALIGN, "norm scratch and norm_sq must be 8-byte aligned");
  const int64_t need = a->nchunks + zk::kNormScratchExtra;
  if (scratch_count < need)
    return fail(ZERO_EINVAL, "norm scratch holds %lld doubles, %lld needed",
                (long long)scratch_count, (long long)need);
  others.push_back({uintptr_t(scratch), uintptr_t(scratch) + uintptr_t(need) * 8,
                    "the norm scratch"});
  others.push_back({uintptr_t(norm_sq), uintptr_t(norm_sq) + 8, "norm_sq"});
  if (int e = check_disjoint(others)) return e;
  a->partials = scratch;
  a->out = norm_sq;
  return ZERO_OK;
}

// A clipped step chained to the norm of `na` (after attach_norm_buffers): the
// norm's total kernel forms the step's multiplier into the scratch slot after
// the partials, and the step reads it there.
void chain_multiplier(zk::NormArgs* na, zk::StepArgs* a) {
  na->gm_out = reinterpret_cast<float*>(na->partials + na->nchunks + 1);
  na->gscale = a->gscale;
  na->max_norm = a->max_norm;
  a->gm_dev = na->gm_out;
}

// The gradients' buffer ranges of a norm pass.
std::vector<Range> grad_ranges(const void* const* grads, int64_t n, int32_t N, int es) {
  std::vector<Range> rs;
  if (n > 0)
    for (int32_t r = 0; r < N; ++r)
      rs.push_back({uintptr_t(grads[r]), uintptr_t(grads[r]) + uintptr_t(n) * es, "a gradient"});
  return rs;
}

}  // namespace

extern "C" {

const char* zero_strerror(int code) {
  switch (code) {
    case ZERO_OK: return "ok";
    case ZERO_EINVAL: return "invalid argument";
    case ZERO_EALIGN: return "misaligned pointer";
    case ZERO_ECUDA: return "CUDA runtime error";
    case ZERO_ETIMEDOUT: return "timed out";
    case ZERO_ENOMEM: return "out of host memory";
    default: return "unknown status code";
  }
}

const char* zero_last_error(void) { return g_last_error; }

int zero_debug_fail_host_allocs(int32_t count) {
  g_failing_allocs = count > 0 ? count : 0;
  return ZERO_OK;
}

int zero_shard_bounds(int64_t n, int32_t N, int64_t* bounds) {
  if (n < 0) return fail(ZERO_EINVAL, "n=%lld must be >= 0", (long long)n);
  if (N < 1) return fail(ZERO_EINVAL, "N=%d must be >= 1", N);
  if (!bounds) return fail(ZERO_EINVAL, "bounds is NULL");
  shard_bounds(n, N, bounds);
  return ZERO_OK;
}

}  // extern "C"

namespace {

// Whole-tensor shards: the tensor list is split like the indices of
// np.array_split, and the shard bounds are the offsets of those tensors.
int tensor_bounds(const int64_t* numels, int64_t T, int32_t N, int64_t* bounds) {
  if (T < 0) return fail(ZERO_EINVAL, "T=%lld must be >= 0", (long long)T);
  if (N < 1) return fail(ZERO_EINVAL, "N=%d must be >= 1", N);
  if (!bounds || (T > 0 && !numels)) return fail(ZERO_EINVAL, "numels or bounds is NULL");
  std::vector<int64_t> first(size_t(N) + 1);
  shard_bounds(T, N, first.data());
  int64_t offset = 0, k = 0;
  for (int32_t i = 0; i <= N; ++i) {
    while (k < first[i]) {
      if (numels[k] < 0) return fail(ZERO_EINVAL, "tensor %lld has a negative size", (long long)k);
      if (offset > INT64_MAX - numels[k]) return fail(ZERO_EINVAL, "tensor sizes overflow");
      offset += numels[k++];
    }
    bounds[i] = offset;
  }
  return ZERO_OK;
}

// Caller-given shard bounds: N+1 offsets rising from 0 to n.
int check_bounds(const int64_t* b, int64_t n, int32_t N) {
  if (b[0] != 0 || b[N] != n) return fail(ZERO_EINVAL, "shard bounds must start at 0 and end at n");
  for (int32_t i = 0; i < N; ++i)
    if (b[i + 1] < b[i]) return fail(ZERO_EINVAL, "shard bounds must not decrease");
  return ZERO_OK;
}

// Model-state bytes of one rank whose shard holds s of the n parameters.
int breakdown(int64_t n, int32_t stage, int32_t precision, uint64_t s, uint64_t out[3]) {
  const uint64_t un = uint64_t(n);
  uint64_t p = 0, g = 0, o = 0;
  bool ok = true;
  if (precision == ZERO_FP64_EMU) {
    // The course's float64 bookkeeping: 8-byte values; stage 1 keeps the full
    // averaged .grad plus the chunk's; stages 1-2 hold m, v and a master chunk;
    // stage 3's chunk is the parameter storage; one process holds m, v of all n.
    ok &= mul_add(8, stage == 3 ? s : un, &p);
    if (stage == 0) ok &= mul_add(8, un, &g);
    else if (stage == 1) ok &= mul_add(8, un, &g) && mul_add(8, s, &g);
    else ok &= mul_add(8, s, &g);
    if (stage == 0) ok &= mul_add(16, un, &o);
    else if (stage == 3) ok &= mul_add(16, s, &o);
    else ok &= mul_add(24, s, &o);
  } else if (precision == ZERO_FP32 || precision == ZERO_BF16_MIXED) {
    const uint64_t P = precision == ZERO_FP32 ? 4 : 2;
    const uint64_t G = P;
    const uint64_t K = precision == ZERO_FP32 ? 8 : 12;
    ok &= mul_add(P, stage == 3 ? s : un, &p);
    ok &= mul_add(G, stage >= 2 ? s : un, &g);
    ok &= mul_add(K, stage >= 1 ? s : un, &o);
  } else {
    return fail(ZERO_EINVAL, "unknown precision %d", precision);
  }
  if (!ok) return fail(ZERO_EINVAL, "byte count overflows 64 bits");
  out[0] = p;
  out[1] = g;
  out[2] = o;
  return ZERO_OK;
}

// The multiplier of the mean gradient and, when max_grad_norm > 0, clipping
// with the squared norm at norm_sq (read on the device; with norm_scratch the
// call writes it there first).
int fill_scale_clip(double grad_scale, double max_grad_norm, const double* norm_sq,
                    zk::StepArgs* a) {
  if (!std::isfinite(grad_scale) || !(grad_scale > 0.0))
    return fail(ZERO_EINVAL, "grad_scale must be finite and > 0");
  a->gscale = grad_scale;
  if (max_grad_norm > 0.0) {
    if (!std::isfinite(max_grad_norm)) return fail(ZERO_EINVAL, "max_grad_norm must be finite");
    if (!norm_sq) return fail(ZERO_EINVAL, "clipping needs the squared norm (norm_sq)");
    a->max_norm = max_grad_norm;
    a->norm_sq = norm_sq;
  }
  return ZERO_OK;
}

// zero_step_opts_t -> StepArgs (after prepare_step).
int fill_adamw(const zero_step_opts_t* o, zk::StepArgs* a) {
  if (int e = adam_consts(o->t, o->lr, o->beta1, o->beta2, o->eps, o->weight_decay, &a->c))
    return e;
  if (int e = fill_scale_clip(o->grad_scale, o->max_grad_norm, o->norm_sq, a)) return e;
  a->owner_only = o->owner_only != 0;
  return ZERO_OK;
}

// Checks zero_sgd_opts_t; the kernel variant it needs.
int sgd_opt(const zero_sgd_opts_t* o, zk::Opt* opt) {
  if (o->t < 1) return fail(ZERO_EINVAL, "step number t=%lld must be >= 1", (long long)o->t);
  if (!std::isfinite(o->lr) || o->lr < 0.0) return fail(ZERO_EINVAL, "lr must be finite and >= 0");
  if (!std::isfinite(o->momentum) || o->momentum < 0.0)
    return fail(ZERO_EINVAL, "momentum must be finite and >= 0");
  if (!std::isfinite(o->dampening)) return fail(ZERO_EINVAL, "dampening must be finite");
  if (!std::isfinite(o->weight_decay)) return fail(ZERO_EINVAL, "weight_decay must be finite");
  if (o->nesterov && (o->momentum <= 0.0 || o->dampening != 0.0))
    return fail(ZERO_EINVAL, "Nesterov momentum needs momentum > 0 and zero dampening");
  *opt = o->momentum != 0.0 ? zk::Opt::SgdMomentum : zk::Opt::Sgd;
  return ZERO_OK;
}

// zero_sgd_opts_t -> StepArgs (after prepare_step).
int fill_sgd(const zero_sgd_opts_t* o, zk::StepArgs* a) {
  a->sgd.lr = float(o->lr);
  a->sgd.wd = float(o->weight_decay);
  a->sgd.mu = float(o->momentum);
  a->sgd.omd = float(1.0 - o->dampening);
  a->sgd.wd_on = o->weight_decay != 0.0;
  a->sgd.first = o->t == 1;
  a->sgd.nesterov = o->nesterov != 0;
  if (int e = fill_scale_clip(o->grad_scale, o->max_grad_norm, o->norm_sq, a)) return e;
  a->owner_only = o->owner_only != 0;
  return ZERO_OK;
}

int check_range(int64_t lo, int64_t hi, int64_t n) {
  if (lo < 0 || hi < lo || hi > n)
    return fail(ZERO_EINVAL, "range [%lld, %lld) outside [0, %lld)", (long long)lo, (long long)hi,
                (long long)n);
  return ZERO_OK;
}

// The step of zero_step_ex / zero_step_sgd over [lo, hi), after the options
// are filled in. With clipping and norm_scratch the call forms the norm
// itself: the partial sums of the whole gradient into the scratch, their
// fixed-order total into norm_sq (the two launches of zero_grad_norm_sq), then
// the step, each launch a programmatic dependent of the one before.
int run_step(zk::StepArgs& a, zero_states* st, const void* const* grads, bool vec, int phase,
             int64_t lo, int64_t hi, double* norm_scratch, int64_t scratch_count,
             const std::vector<Range>& bufs, cudaStream_t s, zk::Opt opt) {
  if (a.norm_sq && norm_scratch) {
    zk::NormArgs na;
    if (int e = prepare_norm(grads, st->n, st->N, st->precision, &na)) return e;
    if (int e = attach_norm_buffers(norm_scratch, scratch_count, const_cast<double*>(a.norm_sq),
                                    bufs, &na))
      return e;
    chain_multiplier(&na, &a);
    cudaError_t ce = zk::launch_norm(na, st->precision == ZERO_BF16_MIXED, s);
    if (ce != cudaSuccess) return cuda_fail(ce, "gradient norm kernel launch");
    a.dependent = 1;
  }
  return launch_range(a, st, vec, phase, lo, hi, s, opt);
}

}  // namespace

extern "C" {

int zero_memory_breakdown(int64_t n, int32_t N, int32_t stage, int32_t precision, int32_t rank,
                          uint64_t out[3]) {
  if (n < 0 || N < 1) return fail(ZERO_EINVAL, "need n >= 0 and N >= 1");
  if (stage < 0 || stage > 3) return fail(ZERO_EINVAL, "stage %d outside 0..3", stage);
  if (rank < 0 || rank >= N) return fail(ZERO_EINVAL, "rank %d outside [0, %d)", rank, N);
  if (!out) return fail(ZERO_EINVAL, "out is NULL");
  const int64_t q = n / N, r = n % N;
  return breakdown(n, stage, precision, uint64_t(q + (rank < r ? 1 : 0)), out);
}

int zero_memory_breakdown_ex(int64_t n, int32_t N, int32_t stage, int32_t precision,
                             int32_t rank, const int64_t* bounds, uint64_t out[3]) {
  if (!bounds) return zero_memory_breakdown(n, N, stage, precision, rank, out);
  if (n < 0 || N < 1) return fail(ZERO_EINVAL, "need n >= 0 and N >= 1");
  if (stage < 0 || stage > 3) return fail(ZERO_EINVAL, "stage %d outside 0..3", stage);
  if (rank < 0 || rank >= N) return fail(ZERO_EINVAL, "rank %d outside [0, %d)", rank, N);
  if (!out) return fail(ZERO_EINVAL, "out is NULL");
  if (int e = check_bounds(bounds, n, N)) return e;
  return breakdown(n, stage, precision, uint64_t(bounds[rank + 1] - bounds[rank]), out);
}

int zero_tensor_shard_bounds(const int64_t* numels, int64_t T, int32_t N, int64_t* bounds) {
  return tensor_bounds(numels, T, N, bounds);
}

int zero_memory_bytes(int64_t n, int32_t N, int32_t stage, int32_t precision, uint64_t* out) {
  if (!out) return fail(ZERO_EINVAL, "out is NULL");
  uint64_t b[3];
  if (int e = zero_memory_breakdown(n, N, stage, precision, 0, b)) return e;
  uint64_t total = 0;
  for (uint64_t x : b) {
    if (total > UINT64_MAX - x) return fail(ZERO_EINVAL, "byte count overflows 64 bits");
    total += x;
  }
  *out = total;
  return ZERO_OK;
}

int zero_init_states(int64_t n, int32_t N, int32_t precision, float* m, float* v, float* master,
                     const float* master_init, zero_stream_t stream, zero_states_t** out) {
  return zero_init_states_ex(n, N, precision, m, v, master, master_init, nullptr, stream, out);
}

int zero_init_states_ex(int64_t n, int32_t N, int32_t precision, float* m, float* v,
                        float* master, const float* master_init, const int64_t* bounds,
                        zero_stream_t stream, zero_states_t** out) {
  if (!out) return fail(ZERO_EINVAL, "out is NULL");
  *out = nullptr;
  if (n < 0) return fail(ZERO_EINVAL, "n=%lld must be >= 0", (long long)n);
  if (!valid_ranks(N)) return fail(ZERO_EINVAL, "N=%d outside [1, %d]", N, ZERO_MAX_RANKS);
  if (bounds)
    if (int e = check_bounds(bounds, n, N)) return e;
  if (precision != ZERO_FP32 && precision != ZERO_BF16_MIXED)
    return fail(ZERO_EINVAL, "state precision must be FP32 or BF16_MIXED");
  // v = NULL: state for momentum SGD (m is its buffer); m = v = NULL: plain SGD.
  if (n > 0 && !m && v) return fail(ZERO_EINVAL, "v without m");
  const bool mixed = precision == ZERO_BF16_MIXED;
  if (mixed && n > 0 && (!master || !master_init))
    return fail(ZERO_EINVAL, "mixed precision needs master and master_init");
  if (!mixed && (master || master_init))
    return fail(ZERO_EINVAL, "fp32 state takes no master buffer");
  int ph = -2;
  bool same = true;
  const float* bufs[4] = {m, v, master, master_init};
  std::vector<Range> rs;
  for (int k = 0; k < (mixed ? 4 : 2); ++k) {
    if (!bufs[k]) continue;  // an absent m or v (SGD state)
    const int q = phase_of(bufs[k], 4);
    if (q < 0) return fail(ZERO_EALIGN, "state buffer not 4-byte aligned");
    if (ph == -2) ph = q;
    else if (ph != q) same = false;
    if (n > 0) rs.push_back({uintptr_t(bufs[k]), uintptr_t(bufs[k]) + uintptr_t(n) * 4, "a state buffer"});
  }
  if (int e = check_disjoint(rs)) return e;
  zero_states* st = new_handle<zero_states>();
  if (!st) return fail(ZERO_ENOMEM, "cannot allocate the state handle");
  st->n = n;
  st->N = N;
  st->precision = precision;
  st->m = m;
  st->v = v;
  st->master = master;
  if (bounds) std::memcpy(st->bounds, bounds, sizeof(int64_t) * (N + 1));
  else shard_bounds(n, N, st->bounds);
  if (n > 0) {
    zk::InitArgs ia{m, v, master, master_init, make_split(0, n, same, ph, 4)};
    cudaError_t e = zk::launch_init(ia, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
      delete st;
      return cuda_fail(e, "state init kernel launch");
    }
  }
  *out = st;
  return ZERO_OK;
}

int zero_free_states(zero_states_t* st) {
  if (st) {
    for (cudaEvent_t e : st->events) cudaEventDestroy(e);
  }
  delete st;
  return ZERO_OK;
}

int zero_states_info(const zero_states_t* st, int64_t* n, int32_t* N, int32_t* precision) {
  if (!st) return fail(ZERO_EINVAL, "state handle is NULL");
  if (n) *n = st->n;
  if (N) *N = st->N;
  if (precision) *precision = st->precision;
  return ZERO_OK;
}

int zero_state_view(const zero_states_t* st, int32_t rank, int64_t* lo, int64_t* hi, float** m,
                    float** v, float** master) {
  if (!st) return fail(ZERO_EINVAL, "state handle is NULL");
  if (rank < 0 || rank >= st->N) return fail(ZERO_EINVAL, "rank %d outside [0, %d)", rank, st->N);
  const int64_t a = st->bounds[rank], b = st->bounds[rank + 1];
  if (lo) *lo = a;
  if (hi) *hi = b;
  if (m) *m = st->m ? st->m + a : nullptr;
  if (v) *v = st->v ? st->v + a : nullptr;
  if (master) *master = st->master ? st->master + a : nullptr;
  return ZERO_OK;
}

int zero_step_range(void* const* params, const void* const* grads, zero_states_t* st, int64_t t,
                    double lr, double beta1, double beta2, double eps, double weight_decay,
                    int64_t lo, int64_t hi, zero_stream_t stream) {
  zk::StepArgs a;
  bool vec = false;
  int phase = 0;
  if (int e = prepare_step(params, grads, st, zk::Opt::AdamW, &a, &vec, &phase)) return e;
  if (lo < 0 || hi < lo || hi > st->n)
    return fail(ZERO_EINVAL, "range [%lld, %lld) outside [0, %lld)", (long long)lo, (long long)hi,
                (long long)st->n);
  if (int e = adam_consts(t, lr, beta1, beta2, eps, weight_decay, &a.c)) return e;
  return launch_range(a, st, vec, phase, lo, hi, reinterpret_cast<cudaStream_t>(stream));
}

int zero_step(void* const* params, const void* const* grads, zero_states_t* st, int64_t t,
              double lr, double beta1, double beta2, double eps, double weight_decay,
              zero_stream_t stream) {
  if (!st) return fail(ZERO_EINVAL, "state handle is NULL");
  return zero_step_range(params, grads, st, t, lr, beta1, beta2, eps, weight_decay, 0, st->n,
                         stream);
}

int zero_step_ex(void* const* params, const void* const* grads, zero_states_t* st,
                 const zero_step_opts_t* o, zero_stream_t stream) {
  if (!st) return fail(ZERO_EINVAL, "state handle is NULL");
  if (!o) return fail(ZERO_EINVAL, "options are NULL");
  zk::StepArgs a;
  bool vec = false;
  int phase = 0;
  std::vector<Range> bufs;
  if (int e = prepare_step(params, grads, st, zk::Opt::AdamW, &a, &vec, &phase, &bufs)) return e;
  const int64_t lo = o->lo, hi = o->hi < 0 ? st->n : o->hi;
  if (int e = check_range(lo, hi, st->n)) return e;
  if (int e = fill_adamw(o, &a)) return e;
  return run_step(a, st, grads, vec, phase, lo, hi, o->norm_scratch, o->norm_scratch_count, bufs,
                  reinterpret_cast<cudaStream_t>(stream), zk::Opt::AdamW);
}

int zero_gather(void* const* params, zero_states_t* st, int64_t lo, int64_t hi,
                zero_stream_t stream) {
  if (!st) return fail(ZERO_EINVAL, "state handle is NULL");
  if (!params) return fail(ZERO_EINVAL, "params array is NULL");
  if (hi < 0) hi = st->n;
  if (lo < 0 || hi < lo || hi > st->n)
    return fail(ZERO_EINVAL, "range [%lld, %lld) outside [0, %lld)", (long long)lo, (long long)hi,
                (long long)st->n);
  const int32_t N = st->N;
  const bool bf16 = st->precision == ZERO_BF16_MIXED;
  const int es = bf16 ? 2 : 4;
  zk::GatherArgs a;
  std::memset(&a, 0, sizeof(a));
  a.N = N;
  std::memcpy(a.bounds, st->bounds, sizeof(int64_t) * (N + 1));
  std::vector<Range> rs;
  int ph = -2;
  bool same = true;
  for (int32_t r = 0; r < N; ++r) {
    if (st->n > 0 && !params[r]) return fail(ZERO_EINVAL, "params[%d] is NULL", r);
    const int q = phase_of(params[r], es);
    if (q < 0) return fail(ZERO_EALIGN, "params[%d] not aligned to %d bytes", r, es);
    if (ph == -2) ph = q;
    else if (ph != q) same = false;
    a.reps[r] = params[r];
    if (st->n > 0)
      rs.push_back({uintptr_t(params[r]), uintptr_t(params[r]) + uintptr_t(st->n) * es,
                    "a parameter replica"});
  }
  if (int e = check_disjoint(rs)) return e;
  if (hi <= lo || N == 1) return ZERO_OK;
  a.sp = make_split(lo, hi, same, ph, bf16 ? 8 : 4);
  cudaError_t e = zk::launch_gather(a, bf16, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "zero_gather kernel launch");
  return ZERO_OK;
}

int zero_step_sgd(void* const* params, const void* const* grads, zero_states_t* st,
                  const zero_sgd_opts_t* o, zero_stream_t stream) {
  if (!st) return fail(ZERO_EINVAL, "state handle is NULL");
  if (!o) return fail(ZERO_EINVAL, "options are NULL");
  zk::Opt opt;
  if (int e = sgd_opt(o, &opt)) return e;
  zk::StepArgs a;
  bool vec = false;
  int phase = 0;
  std::vector<Range> bufs;
  if (int e = prepare_step(params, grads, st, opt, &a, &vec, &phase, &bufs)) return e;
  const int64_t lo = o->lo, hi = o->hi < 0 ? st->n : o->hi;
  if (int e = check_range(lo, hi, st->n)) return e;
  if (int e = fill_sgd(o, &a)) return e;
  return run_step(a, st, grads, vec, phase, lo, hi, o->norm_scratch, o->norm_scratch_count, bufs,
                  reinterpret_cast<cudaStream_t>(stream), opt);
}

int zero_grad_norm_scratch_count(int64_t n, int32_t precision, int64_t* count) {
  if (!count) return fail(ZERO_EINVAL, "count is NULL");
  if (n < 0) return fail(ZERO_EINVAL, "n=%lld must be >= 0", (long long)n);
  if (precision != ZERO_FP32 && precision != ZERO_BF16_MIXED)
    return fail(ZERO_EINVAL, "gradient precision must be FP32 or BF16_MIXED");
  *count = (n + zk::kNormChunk - 1) / zk::kNormChunk + zk::kNormScratchExtra;
  return ZERO_OK;
}

int zero_grad_norm_sq(const void* const* grads, int64_t n, int32_t N, int32_t precision,
                      double* scratch, int64_t scratch_count, double* norm_sq,
                      zero_stream_t stream) {
  zk::NormArgs a;
  if (int e = prepare_norm(grads, n, N, precision, &a)) return e;
  const int es = precision == ZERO_BF16_MIXED ? 2 : 4;
  if (int e = attach_norm_buffers(scratch, scratch_count, norm_sq, grad_ranges(grads, n, N, es),
                                  &a))
    return e;
  cudaError_t e = zk::launch_norm(a, es == 2, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "gradient norm kernel launch");
  return ZERO_OK;
}

int zero_grad_norm_sq_noalloc(const void* const* grads, int64_t n, int32_t N, int32_t precision,
                              double* norm_sq, zero_stream_t stream) {
  zk::NormArgs a;
  if (int e = prepare_norm(grads, n, N, precision, &a)) return e;
  if (!norm_sq) return fail(ZERO_EINVAL, "norm_sq is NULL");
  if (reinterpret_cast<uintptr_t>(norm_sq) % 8) return fail(ZERO_EALIGN, "norm_sq not 8-byte aligned");
  if (n > ZERO_NOALLOC_MAX_N || a.nchunks + 1 > zk::kNoAllocPartials)
    return fail(ZERO_EINVAL,
                "n=%lld exceeds the %lld elements the library's own scratch covers; use "
                "zero_grad_norm_sq with caller-provided scratch",
                (long long)n, (long long)ZERO_NOALLOC_MAX_N);
  const int es = precision == ZERO_BF16_MIXED ? 2 : 4;
  std::vector<Range> rs;
  if (n > 0)
    for (int32_t r = 0; r < N; ++r)
      rs.push_back({uintptr_t(grads[r]), uintptr_t(grads[r]) + uintptr_t(n) * es, "a gradient"});
  rs.push_back({uintptr_t(norm_sq), uintptr_t(norm_sq) + 8, "norm_sq"});
  if (int e = check_disjoint(rs)) return e;
  double* partials = nullptr;
  cudaError_t ce = zk::noalloc_partials(&partials);
  if (ce != cudaSuccess) return cuda_fail(ce, "looking up the library's scratch array");
  a.partials = partials;
  a.out = norm_sq;
  ce = zk::launch_norm(a, es == 2, reinterpret_cast<cudaStream_t>(stream));
  if (ce != cudaSuccess) return cuda_fail(ce, "gradient norm kernel launch");
  return ZERO_OK;
}

int zero_bucket_count(int64_t n, int32_t precision, int64_t bucket_bytes, int64_t* count) {
  if (!count) return fail(ZERO_EINVAL, "count is NULL");
  if (n < 0) return fail(ZERO_EINVAL, "n=%lld must be >= 0", (long long)n);
  int64_t B;
  if (int e = bucket_elems(precision, bucket_bytes, &B)) return e;
  *count = bucket_count_of(n, B);
  return ZERO_OK;
}

int zero_bucket_range(int64_t n, int32_t precision, int64_t bucket_bytes, int64_t k, int64_t* lo,
                      int64_t* hi) {
  if (!lo || !hi) return fail(ZERO_EINVAL, "lo/hi is NULL");
  if (n < 0) return fail(ZERO_EINVAL, "n=%lld must be >= 0", (long long)n);
  int64_t B;
  if (int e = bucket_elems(precision, bucket_bytes, &B)) return e;
  if (k < 0 || k >= bucket_count_of(n, B))
    return fail(ZERO_EINVAL, "bucket %lld outside [0, %lld)", (long long)k,
                (long long)bucket_count_of(n, B));
  bucket_range_of(n, B, k, lo, hi);
  return ZERO_OK;
}

int zero_step_bucket(void* const* params, const void* const* grads, zero_states_t* st, int64_t t,
                     double lr, double beta1, double beta2, double eps, double weight_decay,
                     int64_t bucket_bytes, int64_t k, zero_event_t ready, zero_stream_t side) {
  if (!st) return fail(ZERO_EINVAL, "state handle is NULL");
  int64_t lo, hi;
  if (int e = zero_bucket_range(st->n, st->precision, bucket_bytes, k, &lo, &hi)) return e;
  zk::StepArgs a;
  bool vec = false;
  int phase = 0;
  if (int e = prepare_step(params, grads, st, zk::Opt::AdamW, &a, &vec, &phase)) return e;
  if (int e = adam_consts(t, lr, beta1, beta2, eps, weight_decay, &a.c)) return e;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(side);
  if (ready) {
    cudaError_t ce = cudaStreamWaitEvent(s, reinterpret_cast<cudaEvent_t>(ready), 0);
    if (ce != cudaSuccess) return cuda_fail(ce, "cudaStreamWaitEvent");
  }
  return launch_range(a, st, vec, phase, lo, hi, s);
}

int zero_step_bucketed(void* const* params, const void* const* grads, zero_states_t* st,
                       int64_t t, double lr, double beta1, double beta2, double eps,
                       double weight_decay, int64_t bucket_bytes, const zero_event_t* ready,
                       int64_t n_ready, zero_stream_t side, zero_event_t done,
                       int64_t timeout_ms) {
  if (!st) return fail(ZERO_EINVAL, "state handle is NULL");
  int64_t B;
  if (int e = bucket_elems(st->precision, bucket_bytes, &B)) return e;
  const int64_t count = bucket_count_of(st->n, B);
  if (ready ? n_ready != count : n_ready != 0)
    return fail(ZERO_EINVAL, "need %lld ready events (got %lld%s)", (long long)count,
                (long long)n_ready, ready ? "" : ", array NULL");
  zk::StepArgs a;
  bool vec = false;
  int phase = 0;
  if (int e = prepare_step(params, grads, st, zk::Opt::AdamW, &a, &vec, &phase)) return e;
  if (int e = adam_consts(t, lr, beta1, beta2, eps, weight_decay, &a.c)) return e;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(side);
  for (int64_t k = 0; k < count; ++k) {
    if (ready && ready[k]) {
      cudaError_t ce = cudaStreamWaitEvent(s, reinterpret_cast<cudaEvent_t>(ready[k]), 0);
      if (ce != cudaSuccess) return cuda_fail(ce, "cudaStreamWaitEvent");
    }
    int64_t lo, hi;
    bucket_range_of(st->n, B, k, &lo, &hi);
    // buckets after the first may start while the previous one finishes:
    // their index ranges are disjoint
    a.dependent = k > 0;
    if (int e = launch_range(a, st, vec, phase, lo, hi, s)) return e;
  }
  if (done) {
    cudaError_t ce = cudaEventRecord(reinterpret_cast<cudaEvent_t>(done), s);
    if (ce != cudaSuccess) return cuda_fail(ce, "cudaEventRecord");
  }
  if (timeout_ms < 0) return ZERO_OK;
  // Host-side deadline: poll, never block in the driver, never spin on the GPU.
  const auto deadline = std::chrono::steady_clock::now() + std::chrono::milliseconds(timeout_ms);
  for (;;) {
    cudaError_t q = done ? cudaEventQuery(reinterpret_cast<cudaEvent_t>(done)) : cudaStreamQuery(s);
    if (q == cudaSuccess) return ZERO_OK;
    if (q != cudaErrorNotReady) return cuda_fail(q, "waiting for the bucketed step");
    if (std::chrono::steady_clock::now() >= deadline)
      return fail(ZERO_ETIMEDOUT, "bucketed step not finished after %lld ms", (long long)timeout_ms);
    std::this_thread::sleep_for(std::chrono::microseconds(50));
  }
}

int zero_step_from_host(void* const* params, const void* const* host_grads, void* const* staging,
                        zero_states_t* st, int64_t t, double lr, double beta1, double beta2,
                        double eps, double weight_decay, void* host_params_out,
                        int64_t chunk_bytes, zero_stream_t compute, zero_stream_t h2d,
                        zero_stream_t d2h) {
  zero_step_opts_t o;
  std::memset(&o, 0, sizeof(o));
  o.t = t;
  o.lr = lr;
  o.beta1 = beta1;
  o.beta2 = beta2;
  o.eps = eps;
  o.weight_decay = weight_decay;
  o.grad_scale = 1.0;
  o.hi = -1;
  return zero_step_from_host_ex(params, host_grads, staging, st, &o, nullptr, host_params_out,
                                chunk_bytes, compute, h2d, d2h);
}

int zero_step_from_host_ex(void* const* params, const void* const* host_grads,
                           void* const* staging, zero_states_t* st, const zero_step_opts_t* adamw,
                           const zero_sgd_opts_t* sgd, void* host_params_out, int64_t chunk_bytes,
                           zero_stream_t compute, zero_stream_t h2d, zero_stream_t d2h) {
  if (!st) return fail(ZERO_EINVAL, "state handle is NULL");
  if (!host_grads) return fail(ZERO_EINVAL, "host_grads array is NULL");
  if ((adamw == nullptr) == (sgd == nullptr))
    return fail(ZERO_EINVAL, "give exactly one of the AdamW and the SGD options");
  const int64_t o_lo = adamw ? adamw->lo : sgd->lo, o_hi = adamw ? adamw->hi : sgd->hi;
  const bool clip = (adamw ? adamw->max_grad_norm : sgd->max_grad_norm) > 0.0;
  double* norm_out = const_cast<double*>(adamw ? adamw->norm_sq : sgd->norm_sq);
  double* norm_scratch = adamw ? adamw->norm_scratch : sgd->norm_scratch;
  const int64_t norm_count = adamw ? adamw->norm_scratch_count : sgd->norm_scratch_count;
  if (o_lo != 0 || (o_hi >= 0 && o_hi != st->n))
    return fail(ZERO_EINVAL, "the host-input step covers the whole vector (lo = 0, hi = -1 or n)");
  if (clip && !norm_scratch)
    return fail(ZERO_EINVAL, "clipping in the host-input step needs norm_scratch (the norm's "
                "partial sums)");
  zk::Opt opt = zk::Opt::AdamW;
  if (sgd)
    if (int e = sgd_opt(sgd, &opt)) return e;
  const int32_t N = st->N;
  const int64_t n = st->n;
  for (int32_t r = 0; r < N; ++r)
    if (n > 0 && !host_grads[r]) return fail(ZERO_EINVAL, "host_grads[%d] is NULL", r);
  int64_t B;
  if (int e = bucket_elems(st->precision, chunk_bytes, &B)) return e;
  zk::StepArgs a;
  bool vec = false;
  int phase = 0;
  std::vector<Range> bufs;
  // the staging buffers are the kernel's gradient buffers
  if (int e = prepare_step(params, staging, st, opt, &a, &vec, &phase, &bufs)) return e;
  if (int e = adamw ? fill_adamw(adamw, &a) : fill_sgd(sgd, &a)) return e;
  if (n == 0) return ZERO_OK;
  const size_t es = st->precision == ZERO_BF16_MIXED ? 2 : 4;
  zk::NormArgs na;
  if (clip) {
    // the norm's own checks, before anything is queued; the steps then read
    // the total from norm_sq (one total launch, not one per chunk's step)
    if (int e = prepare_norm(staging, n, N, st->precision, &na)) return e;
    if (int e = attach_norm_buffers(norm_scratch, norm_count, norm_out, bufs, &na)) return e;
    chain_multiplier(&na, &a);
  }
  const int64_t count = (n + B - 1) / B;
  const size_t need = size_t(2 * count + 2);
  while (st->events.size() < need) {
    cudaEvent_t ev;
    cudaError_t ce = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
    if (ce != cudaSuccess) return cuda_fail(ce, "cudaEventCreateWithFlags");
    st->events.push_back(ev);
  }
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(compute);
  cudaStream_t hs = reinterpret_cast<cudaStream_t>(h2d);
  cudaStream_t ds = reinterpret_cast<cudaStream_t>(d2h);
  cudaEvent_t* ev = st->events.data();
  auto ck = [&](cudaError_t ce, const char* what) { return ce == cudaSuccess ? 0 : cuda_fail(ce, what); };
  // Chained: the previous step launches on this handle were the previous call
  // of this kind, with the same chunks and staging buffers. Then the copy of
  // chunk k only has to wait for that call's step on chunk k (event done[k]),
  // and the copies overlap the tail of that call (its last steps and its
  // copies back). Otherwise the copies start after everything already queued
  // on `compute`.
  const bool chained = st->host_launches == st->launches && st->host_B == B &&
                       st->host_staging.size() == size_t(N) &&
                       std::equal(staging, staging + N, st->host_staging.begin());
  if (!chained) {
    if (int e = ck(cudaEventRecord(ev[0], cs), "cudaEventRecord")) return e;
    if (int e = ck(cudaStreamWaitEvent(hs, ev[0], 0), "cudaStreamWaitEvent")) return e;
  }
  auto copy_in = [&](int64_t k) -> int {  // on `h2d`: chunk k of every rank's gradient
    const int64_t lo = k * B, hi = std::min<int64_t>(n, lo + B);
    const size_t off = size_t(lo) * es, bytes = size_t(hi - lo) * es;
    if (chained)  // the previous call's step on this chunk has read its staging
      if (int e = ck(cudaStreamWaitEvent(hs, ev[3 + 2 * k], 0), "cudaStreamWaitEvent")) return e;
    for (int32_t r = 0; r < N; ++r) {
      cudaError_t ce = cudaMemcpyAsync(static_cast<char*>(staging[r]) + off,
                                       static_cast<const char*>(host_grads[r]) + off, bytes,
                                       cudaMemcpyHostToDevice, hs);
      if (ce != cudaSuccess) return cuda_fail(ce, "host-to-device copy of a gradient chunk");
    }
    return ck(cudaEventRecord(ev[2 + 2 * k], hs), "cudaEventRecord");
  };
  auto step_out = [&](int64_t k) -> int {  // on `compute`, then `d2h`: step and copy back
    const int64_t lo = k * B, hi = std::min<int64_t>(n, lo + B);
    cudaEvent_t done = ev[3 + 2 * k];
    if (int e = launch_range(a, st, vec, phase, lo, hi, cs, opt)) return e;
    if (int e = ck(cudaEventRecord(done, cs), "cudaEventRecord")) return e;
    if (!host_params_out) return ZERO_OK;
    if (int e = ck(cudaStreamWaitEvent(ds, done, 0), "cudaStreamWaitEvent")) return e;
    // the chunk from replica 0, or (owner-only) each piece from its owner's replica
    for (int32_t r = 0; r < (a.owner_only ? N : 1); ++r) {
      const int64_t p_lo = a.owner_only ? std::max(lo, st->bounds[r]) : lo;
      const int64_t p_hi = a.owner_only ? std::min(hi, st->bounds[r + 1]) : hi;
      if (p_hi <= p_lo) continue;
      const size_t p_off = size_t(p_lo) * es;
      cudaError_t ce = cudaMemcpyAsync(static_cast<char*>(host_params_out) + p_off,
                                       static_cast<const char*>(params[r]) + p_off,
                                       size_t(p_hi - p_lo) * es, cudaMemcpyDeviceToHost, ds);
      if (ce != cudaSuccess) return cuda_fail(ce, "device-to-host copy of a parameter chunk");
    }
    return ZERO_OK;
  };
  if (!clip) {
    // each chunk is stepped as soon as it has arrived
    for (int64_t k = 0; k < count; ++k) {
      if (int e = copy_in(k)) return e;
      if (int e = ck(cudaStreamWaitEvent(cs, ev[2 + 2 * k], 0), "cudaStreamWaitEvent")) return e;
      if (int e = step_out(k)) return e;
    }
  } else {
    // The global norm needs the whole gradient. Its partial sums cover fixed
    // runs of kNormChunk vector elements after the scalar head, so each run
    // whose elements have all arrived is summed as soon as they have: after
    // chunk k, the runs ending at or before its end (all of them once the
    // vector body is in). The last launch adds the scalar head and tail's
    // partial; then the fixed-order total, then the steps (their copies back
    // overlapping the later steps).
    const bool bf16 = st->precision == ZERO_BF16_MIXED;
    const int V = bf16 ? 8 : 4;
    const int64_t body_lo = na.sp.lo + na.sp.head, body_hi = body_lo + na.sp.nvec * V;
    int64_t c_done = 0;
    for (int64_t k = 0; k < count; ++k) {
      if (int e = copy_in(k)) return e;
      const int64_t hi = std::min<int64_t>(n, (k + 1) * B);
      const int64_t c_ready = k + 1 == count ? na.nchunks + 1
                              : hi >= body_hi ? na.nchunks
                              : hi > body_lo  ? (hi - body_lo) / na.chunk
                                              : 0;
      if (c_ready <= c_done) continue;
      if (int e = ck(cudaStreamWaitEvent(cs, ev[2 + 2 * k], 0), "cudaStreamWaitEvent")) return e;
      zk::NormArgs part = na;
      part.c_begin = c_done;
      part.c_end = c_ready;
      if (int e = ck(zk::launch_norm_partials(part, bf16, cs), "gradient norm kernel launch"))
        return e;
      c_done = c_ready;
    }
    if (int e = ck(cudaStreamWaitEvent(cs, ev[2 + 2 * (count - 1)], 0), "cudaStreamWaitEvent"))
      return e;
    if (int e = ck(zk::launch_norm_total(na, cs), "gradient norm kernel launch")) return e;
    for (int64_t k = 0; k < count; ++k)
      if (int e = step_out(k)) return e;
  }
  if (host_params_out) {
    // `compute` completes only after the last parameter chunk reached the host
    if (int e = ck(cudaEventRecord(ev[1], ds), "cudaEventRecord")) return e;
    if (int e = ck(cudaStreamWaitEvent(cs, ev[1], 0), "cudaStreamWaitEvent")) return e;
  }
  st->host_launches = st->launches;
  st->host_B = B;
  st->host_staging.assign(staging, staging + N);
  return ZERO_OK;
}

int ddp_allreduce_mean(void* const* grads, int64_t n, int32_t N, int32_t precision,
                       zero_stream_t stream) {
  if (n < 0) return fail(ZERO_EINVAL, "n=%lld must be >= 0", (long long)n);
  if (!valid_ranks(N)) return fail(ZERO_EINVAL, "N=%d outside [1, %d]", N, ZERO_MAX_RANKS);
  if (precision != ZERO_FP32 && precision != ZERO_BF16_MIXED)
    return fail(ZERO_EINVAL, "gradient precision must be FP32 or BF16_MIXED");
  if (!grads) return fail(ZERO_EINVAL, "grads array is NULL");
  const int es = precision == ZERO_BF16_MIXED ? 2 : 4;
  zk::AllreduceArgs a;
  std::memset(&a, 0, sizeof(a));
  a.N = N;
  a.fN = float(N);
  int ph = -2;
  bool same = true;
  std::vector<Range> rs;
  for (int32_t r = 0; r < N; ++r) {
    if (n > 0 && !grads[r]) return fail(ZERO_EINVAL, "grads[%d] is NULL", r);
    const int q = phase_of(grads[r], es);
    if (q < 0) return fail(ZERO_EALIGN, "grads[%d] not aligned to %d bytes", r, es);
    if (ph == -2) ph = q;
    else if (ph != q) same = false;
    a.grads[r] = grads[r];
    if (n > 0) rs.push_back({uintptr_t(grads[r]), uintptr_t(grads[r]) + uintptr_t(n) * es, "a gradient"});
  }
  if (int e = check_disjoint(rs)) return e;
  if (n == 0) return ZERO_OK;
  a.sp = make_split(0, n, same, ph, es == 2 ? 8 : 4);
  cudaError_t e = zk::launch_allreduce(a, es == 2, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "ddp_allreduce_mean kernel launch");
  return ZERO_OK;
}

}  // extern "C"

// Chained DDP host-input calls (ddp_allreduce_mean_from_host_h): the events
// of the last call and the configuration they belong to.
struct zero_ddp_host {
  int device = -1;
  std::vector<cudaEvent_t> events;  // [0] start, [1] end, [2+2k] landed k, [3+2k] released k
  bool have_last = false;           // the last call queued completely
  int64_t n = 0, B = 0;
  int32_t N = 0, precision = 0;
  std::vector<void*> staging;
};

namespace {

// Checks of a DDP host-input call, before anything is queued; the chunk size
// in elements.
int ddp_host_checks(const void* const* host_grads, void* const* staging, int64_t n, int32_t N,
                    int32_t precision, int64_t chunk_bytes, zero_stream_t compute, int64_t* B) {
  if (n < 0) return fail(ZERO_EINVAL, "n=%lld must be >= 0", (long long)n);
  if (!valid_ranks(N)) return fail(ZERO_EINVAL, "N=%d outside [1, %d]", N, ZERO_MAX_RANKS);
  if (!host_grads || !staging) return fail(ZERO_EINVAL, "host_grads or staging array is NULL");
  if (int e = bucket_elems(precision, chunk_bytes, B)) return e;
  const size_t es = precision == ZERO_BF16_MIXED ? 2 : 4;
  for (int32_t r = 0; r < N; ++r)
    if (n > 0 && (!host_grads[r] || !staging[r]))
      return fail(ZERO_EINVAL, "host_grads[%d] or staging[%d] is NULL", r, r);
  // the whole-vector checks (alignment, distinct buffers) before anything is queued
  if (int e = ddp_allreduce_mean(staging, 0, N, precision, compute)) return e;
  std::vector<Range> rs;
  for (int32_t r = 0; r < N && n > 0; ++r)
    rs.push_back({uintptr_t(staging[r]), uintptr_t(staging[r]) + uintptr_t(n) * es,
                  "a staging buffer"});
  return check_disjoint(rs);
}

// Grows `pool` to `need` events of the current device.
int grow_events(std::vector<cudaEvent_t>& pool, size_t need) {
  while (pool.size() < need) {
    cudaEvent_t ev;
    cudaError_t ce = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
    if (ce != cudaSuccess) return cuda_fail(ce, "cudaEventCreateWithFlags");
    pool.push_back(ev);
  }
  return ZERO_OK;
}

// The chunk pipeline of the DDP mean from host memory, on events
// ev[0 .. 2 + 2*count). Unchained, the copies start after everything queued
// on `compute`; chained (the previous call on the same events had the same
// buffers and chunks), the copy of chunk k waits only for that call's
// release of chunk k: its mean and its copy back.
int ddp_host_pipeline(cudaEvent_t* ev, bool chained, const void* const* host_grads,
                      void* const* staging, int64_t n, int32_t N, int32_t precision,
                      void* host_mean_out, int64_t B, zero_stream_t compute, zero_stream_t h2d,
                      zero_stream_t d2h) {
  const size_t es = precision == ZERO_BF16_MIXED ? 2 : 4;
  const int64_t count = (n + B - 1) / B;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(compute);
  cudaStream_t hs = reinterpret_cast<cudaStream_t>(h2d);
  cudaStream_t ds = reinterpret_cast<cudaStream_t>(d2h);
  auto ck = [&](cudaError_t ce, const char* what) { return ce == cudaSuccess ? 0 : cuda_fail(ce, what); };
  if (!chained) {  // the copies start after everything already queued on `compute`
    if (int e = ck(cudaEventRecord(ev[0], cs), "cudaEventRecord")) return e;
    if (int e = ck(cudaStreamWaitEvent(hs, ev[0], 0), "cudaStreamWaitEvent")) return e;
    if (host_mean_out)
      if (int e = ck(cudaStreamWaitEvent(ds, ev[0], 0), "cudaStreamWaitEvent")) return e;
  }
  std::vector<void*> chunk(size_t(N), nullptr);
  for (int64_t k = 0; k < count; ++k) {
    const int64_t lo = k * B, hi = std::min<int64_t>(n, lo + B);
    const size_t off = size_t(lo) * es, bytes = size_t(hi - lo) * es;
    cudaEvent_t landed = ev[2 + 2 * k], released = ev[3 + 2 * k];
    if (chained)  // the previous call's mean and copy back of this chunk are done
      if (int e = ck(cudaStreamWaitEvent(hs, released, 0), "cudaStreamWaitEvent")) return e;
    for (int32_t r = 0; r < N; ++r) {
      cudaError_t ce = cudaMemcpyAsync(static_cast<char*>(staging[r]) + off,
                                       static_cast<const char*>(host_grads[r]) + off, bytes,
                                       cudaMemcpyHostToDevice, hs);
      if (ce != cudaSuccess) return cuda_fail(ce, "host-to-device copy of a gradient chunk");
      chunk[size_t(r)] = static_cast<char*>(staging[r]) + off;
    }
    if (int e = ck(cudaEventRecord(landed, hs), "cudaEventRecord")) return e;
    if (int e = ck(cudaStreamWaitEvent(cs, landed, 0), "cudaStreamWaitEvent")) return e;
    if (int e = ddp_allreduce_mean(chunk.data(), hi - lo, N, precision, compute)) return e;
    if (int e = ck(cudaEventRecord(released, cs), "cudaEventRecord")) return e;
    if (host_mean_out) {
      if (int e = ck(cudaStreamWaitEvent(ds, released, 0), "cudaStreamWaitEvent")) return e;
      cudaError_t ce = cudaMemcpyAsync(static_cast<char*>(host_mean_out) + off, chunk[0], bytes,
                                       cudaMemcpyDeviceToHost, ds);
      if (ce != cudaSuccess) return cuda_fail(ce, "device-to-host copy of a mean chunk");
      // released again once the copy back has read the chunk
      if (int e = ck(cudaEventRecord(released, ds), "cudaEventRecord")) return e;
    }
  }
  // `compute` completes only after the last copy in either direction
  if (int e = ck(cudaEventRecord(ev[1], hs), "cudaEventRecord")) return e;
  if (int e = ck(cudaStreamWaitEvent(cs, ev[1], 0), "cudaStreamWaitEvent")) return e;
  if (host_mean_out) {
    if (int e = ck(cudaEventRecord(ev[1], ds), "cudaEventRecord")) return e;
    if (int e = ck(cudaStreamWaitEvent(cs, ev[1], 0), "cudaStreamWaitEvent")) return e;
  }
  return ZERO_OK;
}

}  // namespace

extern "C" {

int ddp_allreduce_mean_from_host(const void* const* host_grads, void* const* staging, int64_t n,
                                 int32_t N, int32_t precision, void* host_mean_out,
                                 int64_t chunk_bytes, zero_stream_t compute, zero_stream_t h2d,
                                 zero_stream_t d2h) {
  int64_t B;
  if (int e = ddp_host_checks(host_grads, staging, n, N, precision, chunk_bytes, compute, &B))
    return e;
  if (n == 0) return ZERO_OK;
  const int64_t count = (n + B - 1) / B;
  // Events come from a process-wide pool per device, grown on demand. A wait
  // takes the state of an event when it is queued, so re-recording an event in
  // a later call is safe; the mutex keeps two host threads from interleaving
  // their record/wait pairs on one event. These calls never chain.
  static std::mutex mu;
  static std::vector<cudaEvent_t> pools[256];
  int dev = 0;
  {
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess) return cuda_fail(ce, "cudaGetDevice");
    if (dev < 0 || dev >= 256) return fail(ZERO_EINVAL, "device %d outside the event pools", dev);
  }
  std::lock_guard<std::mutex> lock(mu);
  std::vector<cudaEvent_t>& pool = pools[dev];
  if (int e = grow_events(pool, size_t(2 + 2 * count))) return e;
  return ddp_host_pipeline(pool.data(), false, host_grads, staging, n, N, precision,
                           host_mean_out, B, compute, h2d, d2h);
}

int zero_ddp_host_create(zero_ddp_host_t** out) {
  if (!out) return fail(ZERO_EINVAL, "out is NULL");
  *out = new_handle<zero_ddp_host>();
  if (!*out) return fail(ZERO_ENOMEM, "cannot allocate the DDP host-input handle");
  return ZERO_OK;
}

int zero_ddp_host_reset(zero_ddp_host_t* h) {
  if (!h) return fail(ZERO_EINVAL, "handle is NULL");
  h->have_last = false;
  return ZERO_OK;
}

int zero_ddp_host_free(zero_ddp_host_t* h) {
  if (h)
    for (cudaEvent_t e : h->events) cudaEventDestroy(e);
  delete h;
  return ZERO_OK;
}

int ddp_allreduce_mean_from_host_h(zero_ddp_host_t* h, const void* const* host_grads,
                                   void* const* staging, int64_t n, int32_t N, int32_t precision,
                                   void* host_mean_out, int64_t chunk_bytes, zero_stream_t compute,
                                   zero_stream_t h2d, zero_stream_t d2h) {
  if (!h) return fail(ZERO_EINVAL, "handle is NULL");
  int64_t B;
  if (int e = ddp_host_checks(host_grads, staging, n, N, precision, chunk_bytes, compute, &B))
    return e;
  if (n == 0) return ZERO_OK;
  int dev = 0;
  {
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess) return cuda_fail(ce, "cudaGetDevice");
  }
  if (h->device >= 0 && h->device != dev)
    return fail(ZERO_EINVAL, "the handle belongs to device %d, not the current device %d",
                h->device, dev);
  const int64_t count = (n + B - 1) / B;
  if (int e = grow_events(h->events, size_t(2 + 2 * count))) return e;
  h->device = dev;
  const bool chained = h->have_last && h->n == n && h->N == N && h->precision == precision &&
                       h->B == B && h->staging.size() == size_t(N) &&
                       std::equal(staging, staging + N, h->staging.begin());
  h->have_last = false;  // until this call has queued completely
  if (int e = ddp_host_pipeline(h->events.data(), chained, host_grads, staging, n, N, precision,
                                host_mean_out, B, compute, h2d, d2h))
    return e;
  h->have_last = true;
  h->n = n;
  h->N = N;
  h->precision = precision;
  h->B = B;
  h->staging.assign(staging, staging + N);
  return ZERO_OK;
}

}  // extern "C"
