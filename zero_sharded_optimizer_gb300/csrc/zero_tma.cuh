// Bulk-copy (TMA) staged kernels: the fused ZeRO step (AdamW or SGD, with the
// all-gather or owner-only) and the DDP mean for N <= 8 ranks. Included by
// zero_kernels.cu after the element helpers.
//
// Pipeline (one CTA per SM, persistent over tiles tile = blockIdx.x + k*gridDim.x):
//   * per tile, one cp.async.bulk global->shared copy per input stream (N
//     gradient tiles, parameter/master, optimizer state) completing on the
//     stage's mbarrier;
//   * the compute threads wait on the stage, compute, and write the results
//     into an output buffer (or back into the stage); then cp.async.bulk
//     shared->global copies store them: state, (master,) and the same
//     parameter tile N times -- the all-gather reads one shared tile N times
//     instead of N register copies;
//   * an input stage is refilled with the tile kStages ahead once it has been
//     computed, and an output buffer is rewritten only after its previous bulk
//     stores have read it (cp.async.bulk.wait_group.read).
// Two drivers run that loop: the lock-step one (every thread computes, thread
// 0 also issues the copies, block barriers between phases) and the
// warp-specialised one (a load warp, a store warp and compute warps handing
// tiles over by mbarriers). Large tiles (2048 elements, 8 KB per fp32 stream)
// give every stream long contiguous DRAM bursts. The pipeline shape (threads,
// stages, output buffers, shared-memory budget) is a template parameter; the
// named shapes below are the measured choices.
//
// Every wait on an mbarrier is bounded by %globaltimer. When the bound runs
// out the CTA sets ZK_STATUS_WAIT_TIMEOUT in the device status word, waits
// (again bounded) for its own copies still in flight, and returns.

#pragma once

namespace zk {

__device__ unsigned int g_device_status = 0;
constexpr unsigned int ZK_STATUS_WAIT_TIMEOUT = 1u;
constexpr uint64_t kDrainNs = 2000000000ull;   // bound of the drain after a timeout

namespace {

// ------------------------------------------------------------- PTX wrappers --

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}
// Wait for phase `parity` of `bar`; false when `limit_ns` passed first.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}
// Bulk copy global -> shared, completing `bytes` on `bar` (16-byte aligned
// addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}
// Bulk copy shared -> global in the current bulk group.
__device__ __forceinline__ void bulk_store(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
               "r"(smem_addr(src)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// All but the most recent bulk group have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all_but_last() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// All but the KEEP most recent bulk groups have finished reading shared memory.
template <int KEEP>
__device__ __forceinline__ void bulk_wait_read_keep() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(KEEP) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Make this thread's generic-proxy shared-memory writes visible to bulk copies.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------ pipeline shape --

// THREADS per CTA, STAGES input stages, OUTBUFS output buffers (0: results are
// written back into the input stage), BUDGET bytes of dynamic shared memory.
template <int THREADS, int STAGES, int OUTBUFS, int BUDGET>
struct PipeCfg {
  static constexpr int kThreads = THREADS;
  static constexpr int kStages = STAGES;
  static constexpr int kOutBufs = OUTBUFS;
  // Tile size: the largest of 2048, 1536, 1024, 512 elements whose input stages
  // (in_bytes per element) and output buffers (out_bytes per element) fit.
  static constexpr int tile(int in_bytes, int out_bytes) {
    return (STAGES * in_bytes + OUTBUFS * out_bytes) * 2048 <= BUDGET   ? 2048
           : (STAGES * in_bytes + OUTBUFS * out_bytes) * 1536 <= BUDGET ? 1536
           : (STAGES * in_bytes + OUTBUFS * out_bytes) * 1024 <= BUDGET ? 1024
                                                                        : 512;
  }
};

using DefaultPipe = PipeCfg<512, 3, 2, 224 * 1024>;
// The same loop computing in place in three stages: for the fp32 step with its
// all-gather when the output buffers would cost tile size (N >= 5) or the range
// is large (see launch_step_tma).
using InPlacePipe = PipeCfg<512, 3, 0, 224 * 1024>;
// Shapes of the warp-specialised pipeline (compute threads, stages, output
// buffers), measured per optimizer. The owner-only AdamW step computes in place
// in three stages (no output buffers, so all of shared memory holds loads):
// 0.253 -> 0.222 ms per stage-3 step on fp32_25m against three stages and two
// output buffers; four in-place stages measured slower. SGD keeps two stages
// and three output buffers (5 % faster than three stages on gpt2_small and
// fp32_320m; its in-place shapes measured 2-6 % slower).
using WsPipeAdamW = PipeCfg<512, 3, 0, 224 * 1024>;
using WsPipeSgd = PipeCfg<512, 2, 3, 224 * 1024>;
// Shape of the DDP mean's lock-step pipeline: three stages computed in place
// (the mean overwrites the first rank's tile, which is then stored N times).
// Measured against 3 stages + 2 output buffers: 0.128 -> 0.1275 ms on fp32_25m,
// 0.622 -> 0.605 ms on gpt2_small; 4 or 5 in-place stages were no better.
using MeanPipe = PipeCfg<512, 3, 0, 224 * 1024>;

// KS fp32 state streams besides the parameter / master (AdamW 2, momentum
// SGD 1, plain SGD 0).
template <int NR, bool MIXED, int KS, class Cfg>
struct StepTile {
  static constexpr int kGB = MIXED ? 2 : 4;                   // gradient / replica bytes
  static constexpr int kF = 1 + KS;                           // fp32 streams per element
  static constexpr int kOutB = 4 * kF + (MIXED ? 2 : 0);      // (+ bf16 replica)
  static constexpr int T = Cfg::tile(NR * kGB + 4 * kF, kOutB);
  static constexpr uint32_t kGradTile = uint32_t(T) * kGB;
  static constexpr uint32_t kFTile = uint32_t(T) * 4;
  static constexpr uint32_t kStage = NR * kGradTile + kF * kFTile;
  static constexpr uint32_t kOut = uint32_t(T) * kOutB;
  static constexpr uint32_t kSmem = Cfg::kStages * kStage + Cfg::kOutBufs * kOut;
};

template <int NR, bool BF16, class Cfg>
struct MeanTile {
  static constexpr int kGB = BF16 ? 2 : 4;
  static constexpr int T = Cfg::tile(NR * kGB, kGB);
  static constexpr uint32_t kTile = uint32_t(T) * kGB;
  static constexpr uint32_t kStage = NR * kTile;
  static constexpr uint32_t kSmem = Cfg::kStages * kStage + Cfg::kOutBufs * kTile;
};

// Elements [a, b) of a shared-memory tile whose first element j0 sits on a
// 16-byte boundary of dst: the 16-byte-aligned middle as one bulk copy, the
// ragged ends (fewer than 16 bytes each) as plain stores by this thread.
template <typename E>
__device__ __forceinline__ void store_slice(E* dst, const E* tile, int64_t j0, int64_t a,
                                            int64_t b) {
  constexpr int64_t U = 16 / int64_t(sizeof(E));
  int64_t a16 = j0 + (a - j0 + U - 1) / U * U;
  int64_t b16 = j0 + (b - j0) / U * U;
  if (a16 >= b16) a16 = b16 = b;  // no aligned middle: all plain stores
  for (int64_t k = a; k < a16; ++k) __stcs(dst + k, tile[k - j0]);
  if (b16 > a16) bulk_store(dst + a16, tile + (a16 - j0), uint32_t((b16 - a16) * sizeof(E)));
  for (int64_t k = b16; k < b; ++k) __stcs(dst + k, tile[k - j0]);
}

// Shared pipeline state of one CTA.
template <int S>
struct PipeState {
  uint64_t full[S];
  int owner[S];  // fp32 step: owner of the whole tile, -1 if it straddles
  int abort;
};

// On a timed-out wait: record it, then wait (bounded) for every tile this CTA
// issued but has not consumed, so no bulk copy writes shared memory after exit.
template <int S>
__device__ __forceinline__ void drain_after_timeout(PipeState<S>& ps, int64_t consumed,
                                                    int64_t issued) {
  atomicOr(&g_device_status, ZK_STATUS_WAIT_TIMEOUT);
  for (int64_t t = consumed; t < issued; ++t)
    mbar_wait(&ps.full[t % S], uint32_t((t / S) & 1), kDrainNs);
}

// A pipeline prologue that does nothing.
struct NoPrologue {
  __device__ __forceinline__ void operator()() const {}
};

// The lock-step loop: every thread computes, thread 0 also issues the copies,
// and block barriers separate the phases. `issue_load(local)` queues the bulk
// loads of local tile `local` into stage local % kStages;
// `compute(local, stage, out)` turns stage `stage` into output
// buffer `out` (or back into the stage when there are no output buffers);
// `issue_store(local, stage, out)` queues and commits the bulk stores of the
// results. `prologue()` runs on every thread once the first loads are issued,
// before the first tile is computed (work that can overlap those loads).
template <class Cfg, typename Load, typename Compute, typename Store,
          typename Prologue = NoPrologue>
__device__ __forceinline__ void run_pipeline(PipeState<Cfg::kStages>& ps, int64_t my_tiles,
                                             uint64_t wait_ns, Load issue_load,
                                             Compute compute, Store issue_store,
                                             Prologue prologue = Prologue()) {
  constexpr int S = Cfg::kStages;
  constexpr int OB = Cfg::kOutBufs > 0 ? Cfg::kOutBufs : 1;
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&ps.full[s], 1);
    fence_mbar_init();
    ps.abort = 0;
  }
  __syncthreads();
  int64_t issued = 0;  // meaningful in thread 0 only
  if (tid == 0) {
    for (; issued < S && issued < my_tiles; ++issued) issue_load(issued);
  }
  prologue();
  for (int64_t k = 0; k < my_tiles; ++k) {
    const int s = int(k % S);
    const int o = int(k % OB);
    if (tid == 0 && !mbar_wait(&ps.full[s], uint32_t((k / S) & 1), wait_ns)) {
      ps.abort = 1;
      drain_after_timeout(ps, k, issued);
    }
    __syncthreads();
    if (ps.abort) break;
    compute(k, s, o);
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      issue_store(k, s, o);
      if constexpr (Cfg::kOutBufs > 0) {
        if (issued < my_tiles) issue_load(issued++);  // into stage s, just consumed
        // the next output buffer (last used OB tiles ago) has been read out
        bulk_wait_read_keep<Cfg::kOutBufs - 1>();
      } else if (k >= 1) {
        bulk_wait_read_all_but_last();  // stores of tile k-1 have read their stage
        if (issued < my_tiles) issue_load(issued++);  // into the stage of tile k-1
      }
    }
  }
  if (tid == 0) bulk_wait_all();
}

// ------------------------------------------------- warp-specialised pipeline --
//
// Thread 0 issues the bulk loads, thread 32 issues the bulk stores, and warps
// 2.. (Cfg::kThreads threads) compute. The roles hand tiles over through
// mbarriers instead of block-wide barriers, so neither the issue of copies nor
// the wait for stores to drain holds up the arithmetic of the next tile.
// With output buffers (OB >= 2):
//   full[s]   the loads of stage s landed           (producer's arrive + bytes)
//   empty[s]  the compute threads are done with s   (one arrival per warp)
//   ready[o]  output buffer o is written            (one arrival per warp)
//   free_[o]  the stores of buffer o have read it   (storer)
// In place (OB == 0: results overwrite the stage, so all of shared memory can
// hold loads):
//   full[s]   as above
//   ready[s]  the results in stage s are written    (one arrival per warp)
//   empty[s]  the stores of stage s have read it    (storer)
// Tile k uses stage k % S and output buffer k % OB; each barrier completes one
// phase per use, so the parity of use u is u & 1.
constexpr int kWsExtraThreads = 64;

template <int S, int OB>
struct PipeStateWS {
  uint64_t full[S];
  uint64_t empty[S];
  uint64_t ready[OB > 0 ? OB : S];
  uint64_t free_[OB > 0 ? OB : 1];  // unused in place
  int owner[S];  // fp32 step: owner of the whole tile, -1 if it straddles
  volatile int abort;
};

// Bounded wait of one role: false when the bound ran out (recorded in the
// device status, and every other role told to stop) or another role stopped.
template <class PS>
__device__ __forceinline__ bool role_wait(PS& ps, uint64_t* bar, uint32_t parity,
                                          uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (ps.abort) return false;
    if (global_timer_ns() - t0 > limit_ns) {
      ps.abort = 1;
      atomicOr(&g_device_status, ZK_STATUS_WAIT_TIMEOUT);
      return false;
    }
  }
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// `issue_load(local)` queues the loads of local tile `local` (arrive.expect_tx
// on full[local % S]); `compute(local, s, o)`, run by the Cfg::kThreads
// compute threads (thread index minus kWsExtraThreads), turns stage s into
// output buffer o; `issue_store(local, s, o)`
// queues and commits the stores of buffer o. `prologue()` runs on the compute
// threads only, before their first tile, while the load warp issues the first
// loads (it may synchronize them with named barrier 1).
template <class Cfg, typename Load, typename Compute, typename Store,
          typename Prologue = NoPrologue>
__device__ __forceinline__ void run_pipeline_ws(PipeStateWS<Cfg::kStages, Cfg::kOutBufs>& ps,
                                                int64_t my_tiles, uint64_t wait_ns,
                                                Load issue_load, Compute compute,
                                                Store issue_store,
                                                Prologue prologue = Prologue()) {
  constexpr int S = Cfg::kStages;
  constexpr int OB = Cfg::kOutBufs;
  constexpr int C = Cfg::kThreads;  // compute threads
  constexpr bool kInPlace = OB == 0;
  static_assert(OB == 0 || OB >= 2, "in place, or at least two output buffers");
  static_assert(C % 32 == 0, "whole compute warps");
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&ps.full[s], 1);
      mbar_init(&ps.empty[s], kInPlace ? 1 : C / 32);
      if constexpr (kInPlace) mbar_init(&ps.ready[s], C / 32);
    }
    for (int o = 0; o < OB; ++o) {
      mbar_init(&ps.ready[o], C / 32);
      mbar_init(&ps.free_[o], 1);
    }
    fence_mbar_init();
    ps.abort = 0;
  }
  __syncthreads();
  // Every loop below exits warp-uniformly (one lane decides and broadcasts,
  // or the lanes vote), so all threads meet the final block barrier converged.
  const int lane = tid & 31, warp = tid >> 5;
  int64_t issued = 0;  // producer lane only
  if (warp == 0) {
    for (int64_t k = 0; k < my_tiles; ++k) {
      const int s = int(k % S);
      int ok = 1;
      if (lane == 0) {
        if (k >= S) ok = role_wait(ps, &ps.empty[s], uint32_t((k / S - 1) & 1), wait_ns);
        if (ok) {
          issue_load(k);
          issued = k + 1;
        }
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
    }
  } else if (warp == 1) {
    for (int64_t k = 0; k < my_tiles; ++k) {
      const int s = int(k % S);
      const int o = kInPlace ? 0 : int(k % (OB > 0 ? OB : 1));
      int ok = 1;
      if (lane == 0) {
        if constexpr (kInPlace) {
          ok = role_wait(ps, &ps.ready[s], uint32_t((k / S) & 1), wait_ns);
          if (ok) {
            issue_store(k, s, o);
            bulk_wait_read_keep<0>();  // the stores have read the stage: reload it
            mbar_arrive(&ps.empty[s]);
          }
        } else {
          ok = role_wait(ps, &ps.ready[o], uint32_t((k / OB) & 1), wait_ns);
          if (ok) {
            issue_store(k, s, o);
            bulk_wait_read_keep<(OB > 0 ? OB - 1 : 0)>();  // tile k - OB + 1 read out
            if (k - OB + 1 >= 0) mbar_arrive(&ps.free_[(k - OB + 1) % OB]);
          }
        }
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
    }
  } else {
    prologue();
    for (int64_t k = 0; k < my_tiles; ++k) {
      const int s = int(k % S);
      const int o = kInPlace ? 0 : int(k % (OB > 0 ? OB : 1));
      int ok = role_wait(ps, &ps.full[s], uint32_t((k / S) & 1), wait_ns);
      if (!kInPlace && ok && k >= OB)
        ok = role_wait(ps, &ps.free_[o], uint32_t((k / (OB > 0 ? OB : 1) - 1) & 1), wait_ns);
      if (!__all_sync(0xffffffffu, ok)) break;
      compute(k, s, o);
      fence_proxy_async_smem();  // this thread's results, seen by the bulk stores
      __syncwarp();              // the warp's reads of stage s and writes are done
      if (lane == 0) {
        if constexpr (kInPlace) {
          mbar_arrive(&ps.ready[s]);
        } else {
          mbar_arrive(&ps.empty[s]);
          mbar_arrive(&ps.ready[o]);
        }
      }
    }
  }
  __syncthreads();
  if (tid == 32) bulk_wait_all();  // every store has finished
  if (tid == 0 && ps.abort) {
    // wait (bounded) for the loads still in flight: the last S issued tiles
    for (int64_t t = issued > S ? issued - S : 0; t < issued; ++t)
      mbar_wait(&ps.full[t % S], uint32_t((t / S) & 1), kDrainNs);
  }
}

// ------------------------------------------------------------ the fused step --

// WS: the warp-specialised pipeline (Cfg::kThreads + kWsExtraThreads threads)
// instead of the lock-step one (Cfg::kThreads threads). NORM: the launch forms
// the clip multiplier from the partial sums of the norm pass launched just
// before it (P.norm_partials): the multiplier is then computed in the
// pipeline's prologue, while the first loads are in flight, and the scalar
// head and tail run after the tiles. Without NORM the multiplier comes first
// (from P.norm_sq, if any); keeping the two apart measured 0.3-0.8 % faster
// for the plain step than one kernel serving both.
template <int NR, bool MIXED, Opt O, bool WS, class Cfg = DefaultPipe, bool NORM = false>
__global__ void __launch_bounds__(Cfg::kThreads + (WS ? kWsExtraThreads : 0), 1)
    zero_step_tma_kernel(const __grid_constant__ StepArgs P) {
  constexpr int KS = kStates<O>;
  using G = StepTile<NR, MIXED, KS, Cfg>;
  constexpr int T = G::T;
  constexpr int V = MIXED ? 8 : 4;
  constexpr int S = Cfg::kStages;
  constexpr int TH = Cfg::kThreads;  // compute threads
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ typename std::conditional<WS, PipeStateWS<S, Cfg::kOutBufs>, PipeState<S>>::type ps;
  const int tid = threadIdx.x;
  // compute-thread index, derived here from threadIdx.x: with its range known
  // and a compile-time stride the compute loop is resolved at compile time
  // (a runtime index or stride measured 1-2 % slower on the whole step)
  const int ct = WS ? tid - kWsExtraThreads : tid;
  const Split& sp = P.sp;
  // Without NORM: the multiplier now (from P.norm_sq, or none).
  float gm = NORM ? 1.0f : grad_multiplier(P);
  // Buckets of one step touch disjoint indices: the next one may start now.
  // This kernel still completes only after the one before it (the wait at the
  // end), so completion on the stream keeps its order.
  pdl_allow_next();

  // Scalar head and tail (fewer than 2V elements) by block 0: first, or with
  // NORM after the tiles, once the multiplier is known.
  auto head_and_tail = [&](int first, int stride, float g_m) {
    if (blockIdx.x != 0) return;
    const int64_t nscalar = sp.head + sp.tail;
    const int64_t body_end = sp.lo + sp.head + sp.nvec * V;
    int owner = 0;
    for (int64_t s = first; s < nscalar; s += stride) {
      const int64_t j = s < sp.head ? sp.lo + s : body_end + (s - sp.head);
      owner = advance_owner(P, owner, j);
      step_scalar<NR, MIXED, O>(P, j, owner, g_m);
    }
  };
  if constexpr (!NORM) head_and_tail(tid, blockDim.x, gm);

  const int64_t base = sp.lo + sp.head;
  const int64_t nelem = sp.nvec * V;
  const int64_t ntiles = (nelem + T - 1) / T;
  const int64_t my_tiles =
      ntiles > int64_t(blockIdx.x) ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  if (my_tiles == 0) {
    if constexpr (NORM) head_and_tail(tid, blockDim.x, group_grad_multiplier(P, tid, blockDim.x, 0));
    pdl_wait_previous();
    return;
  }
  // With NORM, set by the pipeline's prologue in every thread that computes:
  // in the lock-step loop all threads (block barrier), in the
  // warp-specialised loop the compute warps (named barrier 1), while the
  // first loads are in flight.
  auto prologue = [&]() {
    if constexpr (NORM)
      gm = WS ? group_grad_multiplier(P, ct, TH, 1) : group_grad_multiplier(P, tid, blockDim.x, 0);
  };

  auto stage = [&](int s) { return smem + size_t(s) * G::kStage; };
  auto grad_slot = [&](int s, int r) { return stage(s) + r * G::kGradTile; };
  auto in_f = [&](int s, int k) {  // 0 = parameter / master, 1.. = state streams (m, v)
    return reinterpret_cast<float*>(stage(s) + NR * G::kGradTile + k * G::kFTile);
  };
  auto out_f = [&](int s, int o, int k) {
    if constexpr (Cfg::kOutBufs == 0) return in_f(s, k);
    return reinterpret_cast<float*>(smem + S * G::kStage + o * G::kOut + k * G::kFTile);
  };
  auto out_bf = [&](int s, int o) {  // mixed: the bf16 replica tile
    if constexpr (Cfg::kOutBufs == 0) return grad_slot(s, 0);  // consumed gradient slot
    return smem + S * G::kStage + o * G::kOut + G::kF * G::kFTile;
  };
  auto tile_j0 = [&](int64_t local) { return base + (blockIdx.x + local * gridDim.x) * T; };
  auto tile_cnt = [&](int64_t local) {
    const int64_t rem = nelem - (blockIdx.x + local * gridDim.x) * int64_t(T);
    return uint32_t(rem < T ? rem : T);
  };

  auto issue_load = [&](int64_t local) {
    const int s = int(local % S);
    const int64_t j0 = tile_j0(local);
    const uint32_t cnt = tile_cnt(local);
    const uint32_t gbytes = cnt * G::kGB, fbytes = cnt * 4;
    bool straddle = false;
    int owner = 0;
    if constexpr (!MIXED) {
      owner = advance_owner(P, 0, j0);
      straddle = j0 + cnt - 1 >= P.bounds[owner + 1];
      ps.owner[s] = straddle ? -1 : owner;
    }
    mbar_expect_tx(&ps.full[s], NR * gbytes + uint32_t(straddle ? KS : KS + 1) * fbytes);
#pragma unroll
    for (int r = 0; r < NR; ++r)
      bulk_load(grad_slot(s, r), static_cast<const unsigned char*>(P.grads[r]) + j0 * G::kGB,
                gbytes, &ps.full[s]);
    if constexpr (MIXED) {
      bulk_load(in_f(s, 0), P.master + j0, fbytes, &ps.full[s]);
    } else {
      if (!straddle)
        bulk_load(in_f(s, 0), static_cast<const float*>(P.reps[owner]) + j0, fbytes,
                  &ps.full[s]);
    }
#pragma unroll
    for (int k = 0; k < KS; ++k) bulk_load(in_f(s, k + 1), state_ptr(P, k) + j0, fbytes, &ps.full[s]);
  };

  auto issue_store = [&](int64_t local, int s, int o) {
    const int64_t j0 = tile_j0(local);
    const uint32_t cnt = tile_cnt(local);
    const uint32_t fbytes = cnt * 4;
#pragma unroll
    for (int k = 0; k < KS; ++k) bulk_store(state_ptr(P, k) + j0, out_f(s, o, k + 1), fbytes);
    if constexpr (MIXED) bulk_store(P.master + j0, out_f(s, o, 0), fbytes);
    if (P.owner_only) {  // stage 3: each owner's slice of its own replica only
      const int r_lo = advance_owner(P, 0, j0);
      const int r_hi = advance_owner(P, r_lo, j0 + cnt - 1);
      for (int r = r_lo; r <= r_hi; ++r) {
        const int64_t a = j0 > P.bounds[r] ? j0 : P.bounds[r];
        const int64_t b = j0 + cnt < P.bounds[r + 1] ? j0 + cnt : P.bounds[r + 1];
        if constexpr (MIXED)
          store_slice(static_cast<uint16_t*>(P.reps[r]),
                      reinterpret_cast<const uint16_t*>(out_bf(s, o)), j0, a, b);
        else
          store_slice(static_cast<float*>(P.reps[r]), out_f(s, o, 0), j0, a, b);
      }
    } else if constexpr (MIXED) {
#pragma unroll
      for (int r = 0; r < NR; ++r)
        bulk_store(static_cast<unsigned char*>(P.reps[r]) + j0 * 2, out_bf(s, o), cnt * 2);
    } else {
#pragma unroll
      for (int r = 0; r < NR; ++r)
        bulk_store(static_cast<float*>(P.reps[r]) + j0, out_f(s, o, 0), fbytes);
    }
    bulk_commit();
  };

  auto compute = [&](int64_t local, int s, int o) {
    const int64_t j0 = tile_j0(local);
    const int cnt = int(tile_cnt(local));
    const float* pi = in_f(s, 0);
    float* po = out_f(s, o, 0);
    const float* si[kSA<O>];
    float* so[kSA<O>];
#pragma unroll
    for (int k = 0; k < KS; ++k) {
      si[k] = in_f(s, k + 1);
      so[k] = out_f(s, o, k + 1);
    }
    // four elements per thread: float4s of fp32, or one uint2 of bf16 per rank
    for (int q = ct * 4; q < cnt; q += TH * 4) {
      float4 g;
      if constexpr (MIXED) {
        g = unpack4(*reinterpret_cast<const uint2*>(grad_slot(s, 0) + q * 2));
#pragma unroll
        for (int r = 1; r < NR; ++r) {
          const float4 h = unpack4(*reinterpret_cast<const uint2*>(grad_slot(s, r) + q * 2));
          g.x = __fadd_rn(g.x, h.x); g.y = __fadd_rn(g.y, h.y);
          g.z = __fadd_rn(g.z, h.z); g.w = __fadd_rn(g.w, h.w);
        }
      } else {
        g = *reinterpret_cast<const float4*>(grad_slot(s, 0) + q * 4);
#pragma unroll
        for (int r = 1; r < NR; ++r) {
          const float4 h = *reinterpret_cast<const float4*>(grad_slot(s, r) + q * 4);
          g.x = __fadd_rn(g.x, h.x); g.y = __fadd_rn(g.y, h.y);
          g.z = __fadd_rn(g.z, h.z); g.w = __fadd_rn(g.w, h.w);
        }
      }
      float4 p;
      if (MIXED || ps.owner[s] >= 0) {
        p = *reinterpret_cast<const float4*>(pi + q);
      } else {  // the fp32 tile straddles a shard boundary: per-element owners
        float e[4];
        int ow = 0;
        for (int i = 0; i < 4; ++i) {
          ow = advance_owner(P, ow, j0 + q + i);
          e[i] = __ldcs(static_cast<const float*>(P.reps[ow]) + j0 + q + i);
        }
        p = make_float4(e[0], e[1], e[2], e[3]);
      }
      float4 st[kSA<O>];
#pragma unroll
      for (int k = 0; k < KS; ++k) st[k] = *reinterpret_cast<const float4*>(si[k] + q);
      update4<NR, O>(P, gm, g, p, st);
      *reinterpret_cast<float4*>(po + q) = p;
#pragma unroll
      for (int k = 0; k < KS; ++k) *reinterpret_cast<float4*>(so[k] + q) = st[k];
      // in place, this thread's own 8 bytes of the consumed gradient slot
      if constexpr (MIXED) *reinterpret_cast<uint2*>(out_bf(s, o) + q * 2) = pack4(p);
    }
  };

  if constexpr (WS) {
    if constexpr (NORM) {
      run_pipeline_ws<Cfg>(ps, my_tiles, P.wait_ns, issue_load, compute, issue_store, prologue);
      if (ct >= 0) head_and_tail(ct, TH, gm);
    } else {
      run_pipeline_ws<Cfg>(ps, my_tiles, P.wait_ns, issue_load, compute, issue_store);
    }
  } else {
    if constexpr (NORM) {
      run_pipeline<Cfg>(ps, my_tiles, P.wait_ns, issue_load, compute, issue_store, prologue);
      head_and_tail(tid, blockDim.x, gm);
    } else {
      run_pipeline<Cfg>(ps, my_tiles, P.wait_ns, issue_load, compute, issue_store);
    }
  }
  pdl_wait_previous();
}

// ---------------------------------------------------------- the DDP mean --

template <int NR, bool BF16, class Cfg = MeanPipe>
__global__ void __launch_bounds__(Cfg::kThreads, 1)
    allreduce_mean_tma_kernel(const __grid_constant__ AllreduceArgs P) {
  using G = MeanTile<NR, BF16, Cfg>;
  constexpr int T = G::T;
  constexpr int V = BF16 ? 8 : 4;
  constexpr int S = Cfg::kStages;
  constexpr int TH = Cfg::kThreads;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ PipeState<S> ps;
  const int tid = threadIdx.x;
  const Split& sp = P.sp;

  if (blockIdx.x == 0) {
    const int64_t nscalar = sp.head + sp.tail;
    const int64_t body_end = sp.lo + sp.head + sp.nvec * V;
    for (int64_t s = tid; s < nscalar; s += blockDim.x) {
      const int64_t j = s < sp.head ? sp.lo + s : body_end + (s - sp.head);
      mean_scalar<NR, BF16>(P, j);
    }
  }

  const int64_t base = sp.lo + sp.head;
  const int64_t nelem = sp.nvec * V;
  const int64_t ntiles = (nelem + T - 1) / T;
  const int64_t my_tiles =
      ntiles > int64_t(blockIdx.x) ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  if (my_tiles == 0) return;

  auto slot = [&](int s, int r) { return smem + size_t(s) * G::kStage + r * G::kTile; };
  auto out = [&](int s, int o) {
    if constexpr (Cfg::kOutBufs == 0) return slot(s, 0);
    return smem + size_t(S) * G::kStage + o * G::kTile;
  };
  auto tile_j0 = [&](int64_t local) { return base + (blockIdx.x + local * gridDim.x) * T; };
  auto tile_cnt = [&](int64_t local) {
    const int64_t rem = nelem - (blockIdx.x + local * gridDim.x) * int64_t(T);
    return uint32_t(rem < T ? rem : T);
  };
  auto issue_load = [&](int64_t local) {
    const int s = int(local % S);
    const int64_t j0 = tile_j0(local);
    const uint32_t bytes = tile_cnt(local) * G::kGB;
    mbar_expect_tx(&ps.full[s], NR * bytes);
#pragma unroll
    for (int r = 0; r < NR; ++r)
      bulk_load(slot(s, r), static_cast<const unsigned char*>(P.grads[r]) + j0 * G::kGB, bytes,
                &ps.full[s]);
  };
  auto issue_store = [&](int64_t local, int s, int o) {
    const int64_t j0 = tile_j0(local);
    const uint32_t bytes = tile_cnt(local) * G::kGB;
#pragma unroll
    for (int r = 0; r < NR; ++r)
      bulk_store(static_cast<unsigned char*>(P.grads[r]) + j0 * G::kGB, out(s, o), bytes);
    bulk_commit();
  };
  auto compute = [&](int64_t local, int s, int o) {
    const int cnt = int(tile_cnt(local));
    for (int q = tid * 4; q < cnt; q += TH * 4) {
      float4 g;
      if constexpr (BF16) {
        g = unpack4(*reinterpret_cast<const uint2*>(slot(s, 0) + q * 2));
#pragma unroll
        for (int r = 1; r < NR; ++r) {
          const float4 h = unpack4(*reinterpret_cast<const uint2*>(slot(s, r) + q * 2));
          g.x = __fadd_rn(g.x, h.x); g.y = __fadd_rn(g.y, h.y);
          g.z = __fadd_rn(g.z, h.z); g.w = __fadd_rn(g.w, h.w);
        }
      } else {
        g = *reinterpret_cast<const float4*>(slot(s, 0) + q * 4);
#pragma unroll
        for (int r = 1; r < NR; ++r) {
          const float4 h = *reinterpret_cast<const float4*>(slot(s, r) + q * 4);
          g.x = __fadd_rn(g.x, h.x); g.y = __fadd_rn(g.y, h.y);
          g.z = __fadd_rn(g.z, h.z); g.w = __fadd_rn(g.w, h.w);
        }
      }
      g.x = mean_of<NR>(g.x, P.fN); g.y = mean_of<NR>(g.y, P.fN);
      g.z = mean_of<NR>(g.z, P.fN); g.w = mean_of<NR>(g.w, P.fN);
      if constexpr (BF16) {
        *reinterpret_cast<uint2*>(out(s, o) + q * 2) = pack4(g);
      } else {
        *reinterpret_cast<float4*>(out(s, o) + q * 4) = g;
      }
    }
  };
  run_pipeline<Cfg>(ps, my_tiles, P.wait_ns, issue_load, compute, issue_store);
}

}  // namespace
}  // namespace zk
