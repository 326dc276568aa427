// Device helpers and internal launch interface shared by the libpkv sources.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "pkv.h"

namespace pkv {

// Bits of the sticky device error word.
enum : int {
  kErrIndex = 1,     // slot / block id / packed row outside its range
  kErrCapacity = 2,  // sequence longer than its table row, or bad offset / length
  kErrTimeout = 4,   // a bounded mbarrier wait gave up
};

// Default bound on one wait, in nanoseconds of %globaltimer.  A healthy wait
// in these kernels lasts microseconds; this only ends a wait that can never
// complete.  The host may set a shorter bound (pkv_set_wait_limit_ns).
constexpr unsigned long long kWaitTimeoutNs = 4000000000ull;

// A wait looks at its launch's abort word only once it has lasted this long:
// healthy waits end well before, so they never pay for that global load.
constexpr unsigned long long kAbortCheckNs = 100000ull;

__device__ __forceinline__ void set_error(int* err, int bits) {
  if (err) atomicOr(err, bits);
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier (shared::cta) -------------------------------------------------

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// CL: acquire at cluster scope, for a barrier that CTAs of the cluster other
// than this one arrive at (their writes before the arrive become visible).
template <bool CL = false>
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  if constexpr (CL) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
  }
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// The same with an explicit suspend-time hint: the waiting thread sleeps until
// the phase completes or about `hint_ns` pass, instead of polling, so a waiting
// warp takes no issue slots from the warps that work beside it.
template <bool CL = false>
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity,
                                                    uint32_t hint_ns) {
  uint32_t ok;
  if constexpr (CL) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
  }
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// How the waits of one kernel launch give up.  Each wait is bounded by
// limit_ns.  Besides, once any wait of the launch has given up, every other
// pending wait of that launch leaves within a few polls, so a stuck launch
// costs about one bound, not one per CTA and wait.  The signal is the abort
// word that follows the sticky error word in device memory (err[1]): the wait
// that gives up stores its launch's number there (`epoch`, distinct and
// nonzero for every launch the host makes), and the others compare it with
// their own.  A launch therefore never reacts to an earlier launch's give-up.
struct WaitCtl {
  int* err;
  unsigned long long limit_ns;
  int epoch;
};

__device__ __forceinline__ int ld_volatile(const int* p) {
  int v;
  asm volatile("ld.volatile.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ WaitCtl make_wait_ctl(int* err, unsigned long long limit_ns,
                                                 int epoch) {
  WaitCtl w;
  w.err = err;
  w.limit_ns = limit_ns ? limit_ns : kWaitTimeoutNs;
  w.epoch = epoch;
  return w;
}

// True once another wait of this launch has given up.
__device__ __forceinline__ bool launch_gave_up(const WaitCtl& w) {
  return w.err != nullptr && w.epoch != 0 && ld_volatile(w.err + 1) == w.epoch;
}

// Record a give-up: the sticky timeout bit, and this launch's number in the
// abort word so the launch's other waits leave too.
__device__ __forceinline__ void give_up(const WaitCtl& w) {
  if (w.err == nullptr) return;
  atomicOr(w.err, kErrTimeout);
  if (w.epoch != 0) atomicExch(w.err + 1, w.epoch);
}

// The slow part of a wait, entered only after kAbortCheckNs: the bound, the
// launch's abort word, and the give-up.  Kept out of line so the tight poll
// of the healthy case stays as short as a plain one.
template <bool CL = false>
static __device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity,
                                                   const WaitCtl w, unsigned long long t0,
                                                   uint32_t hint_ns) {
#pragma unroll 1
  for (uint32_t it = 1; it < (1u << 30); ++it) {
    if (hint_ns ? mbar_try_wait_sleep<CL>(bar, parity, hint_ns) : mbar_try_wait<CL>(bar, parity))
      return true;
    if (hint_ns || (it & 63u) == 0) {
      if (global_timer_ns() - t0 > w.limit_ns) break;
      if (launch_gave_up(w)) return false;
    }
  }
  give_up(w);
  return false;
}

// Wait for the phase of parity `parity` to complete.  On giving up (bound
// reached, or the launch gave up elsewhere) returns false, the first with
// kErrTimeout set, so the caller can leave cleanly.  Polls: for the short
// waits of the streaming kernels.
template <bool CL = false>
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const WaitCtl& w) {
  if (mbar_try_wait<CL>(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
#pragma unroll 1
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait<CL>(bar, parity)) return true;
    if ((it & 63u) == 0 && global_timer_ns() - t0 > kAbortCheckNs) break;
  }
  return mbar_wait_slow<CL>(bar, parity, w, t0, 0);
}

// The same, sleeping between checks (suspend-time hint): for waits that last
// as long as a tensor-core product, where a polling warp would take issue
// slots from the warp working beside it.
template <bool CL = false>
__device__ __forceinline__ bool mbar_wait_sleep(uint32_t bar, uint32_t parity, const WaitCtl& w) {
  if (mbar_try_wait<CL>(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
#pragma unroll 1
  for (;;) {
    if (mbar_try_wait_sleep<CL>(bar, parity, 20000u)) return true;
    if (global_timer_ns() - t0 > kAbortCheckNs) break;
  }
  return mbar_wait_slow<CL>(bar, parity, w, t0, w.limit_ns < 1000000ull ? 1000u : 100000u);
}

// Wait for asynchronous copies this CTA issued to land before it leaves (or
// re-arms their stage).  Copies complete whatever the other warps do, so this
// wait ignores the launch's give-up and keeps the default bound.
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity, int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
#pragma unroll 1
  for (uint32_t it = 1; it < (1u << 30); ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0 && global_timer_ns() - t0 > kWaitTimeoutNs) break;
  }
  set_error(err, kErrTimeout);
  return false;
}

// ---- bulk (TMA, non-tensor) copy global -> shared ---------------------------
// dst and src 16-byte aligned, bytes a multiple of 16; completion is counted
// on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Orders this thread's earlier generic-proxy global writes before later
// async-proxy (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// ---- programmatic dependent launch -------------------------------------------
// Every kernel of the library starts with griddep_wait(): when it was launched
// as a programmatic dependent, this waits until the grids before it on the
// stream have completed and their memory is visible (a no-op otherwise).  It
// then lets its own dependents launch early; they wait the same way.
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- element conversion ------------------------------------------------------
// bf16 is the upper half of an IEEE fp32 word, so widening is a shift.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Two fp32 values to one bf16 pair (lo in the low half), each rounded to
// nearest even: one packed conversion instruction.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// ---- 16-byte global accesses ------------------------------------------------
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ void st_global(void* p, const uint4& v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

}  // namespace pkv

// ---- internal launch interface (host side, C++ linkage) ---------------------
namespace pkv {

// Launch `kern` on `s`; with `pdl` as a programmatic dependent of the work
// before it (the kernel must call griddep_wait() before reading inputs).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t s, bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

struct PoolView {
  const char* k;  // k_cache bytes
  const char* v;
  char* k_mut;
  char* v_mut;
  long long num_blocks;
  int num_layers;
  int block_size;
  int num_kv_heads;
  int head_dim;
  int elem_size;  // bytes of one stored element (1 for the int8 codes)
  int row_bytes;  // bytes of one token row (int8 pools: codes, scales, padding)
  int quant;      // 1 for int8 pools
  int io_size;    // element size of q, out, k_new, v_new (bf16 for int8 pools)
  int scale_off;  // int8 pools: byte offset of the fp32 scales in a row
};

// Geometry and pointer checks of a pool descriptor (pkv_status value); fills
// `v` when it returns PKV_OK.  `need_ptrs` also checks the two tensors.
int pool_view(const pkv_pool* p, bool need_ptrs, PoolView* v);

cudaError_t launch_slot_mapping(const PoolView& p, const int32_t* bt, int mb, const int32_t* offs,
                                int batch, const int32_t* tok_seq, const int32_t* tok_pos,
                                long long n, int64_t* slots, int* err, cudaStream_t s);

cudaError_t launch_write_slots(const PoolView& p, int layer, const void* k_new, const void* v_new,
                               const int64_t* slots, long long n, int* err, int sm_count,
                               cudaStream_t s);

// Slot mapping and scatter in one kernel (pkv_append_tokens); slots_out may be null.
cudaError_t launch_append(const PoolView& p, int layer, const int32_t* bt, int mb,
                          const int32_t* offs, int batch, const int32_t* tok_seq,
                          const int32_t* tok_pos, long long n, const void* k_new,
                          const void* v_new, int64_t* slots_out, int* err, cudaStream_t s);

cudaError_t launch_gather(const PoolView& p, int layer, const int32_t* bt, int mb,
                          const int32_t* offs, int batch, const int64_t* cu, long long total,
                          void* k_out, void* v_out, int* err, cudaStream_t s);

cudaError_t launch_validate_tables(const PoolView& p, const int32_t* bt, int mb,
                                   const int32_t* lens, const int32_t* offs, int batch,
                                   const int64_t* cu, long long total, int* err, cudaStream_t s);

cudaError_t launch_validate_slots(const PoolView& p, const int64_t* slots, long long n, int* err,
                                  cudaStream_t s);

// Shared-prefix decode: row 0 holds prefix_blocks valid block ids, and every
// table agrees with row 0 on those of them it spans (kErrIndex otherwise).
cudaError_t launch_validate_prefix(const PoolView& p, const int32_t* bt, int mb,
                                   const int32_t* lens, const int32_t* offs, int batch,
                                   int prefix_blocks, int* err, cudaStream_t s);

cudaError_t launch_validate_tokens(const PoolView& p, const int32_t* bt, int mb,
                                   const int32_t* offs, int batch, const int32_t* tok_seq,
                                   const int32_t* tok_pos, long long n, int* err, cudaStream_t s);

struct DecodeLaunch {
  PoolView pool;
  int layer;
  const void* q;
  void* out;
  int num_q_heads;
  float scale;
  const int32_t* bt;
  int mb;
  const int32_t* lens;
  const int32_t* offs;
  int batch;  // <= kDecodeMaxBatch
  void* workspace;
  int grid;  // CTAs of the partial pass
  int* err;
  int smem_optin;  // max dynamic shared memory per block on this device
  cudaEvent_t ev_start = nullptr;  // recorded right before the partial kernel
  cudaEvent_t ev_stop = nullptr;   // recorded right after it
  // fused decode step: the new K / V row of each sequence ([batch] rows of
  // row_bytes), stored at its last position before it is attended to
  const char* k_new = nullptr;
  const char* v_new = nullptr;
  // shared-prefix decode: > 0 runs the suffix pass over the table entries
  // after the first prefix_blocks ones, and leaves the combine to
  // launch_decode_combine_prefix
  int prefix_blocks = 0;
};

constexpr int kDecodeMaxBatch = 2048;

size_t decode_workspace_bytes(int batch, int num_q_heads, int head_dim, int grid);
// 0 = ok; 1 = unsupported shape
int decode_supported(const PoolView& p, int num_q_heads);
cudaError_t launch_decode(const DecodeLaunch& a, cudaStream_t s);
// Shared-prefix decode, after the suffix pass (launch_decode with
// prefix_blocks > 0) and the prefix pass: merge the prefix states
// (pre_ml [nsplit, batch, hq, 2], pre_acc [nsplit, batch, hq, D], fp32) with
// the suffix segments in a.workspace and write a.out (bf16).
cudaError_t launch_decode_combine_prefix(const DecodeLaunch& a, const float* pre_ml,
                                         const float* pre_acc, int nsplit, cudaStream_t s);

// 0 = the prefill kernel handles this pool and head count; 1 = unsupported
int prefill_supported(const PoolView& pv, int num_q_heads);
cudaError_t launch_prefill(const PoolView& pv, int layer, const void* q, int num_q_heads,
                           float scale, const int32_t* bt, int mb, const int32_t* lens,
                           const int32_t* offs, const int64_t* cu_q, int batch, long long total_q,
                           int max_q_len, void* out, int* err, int sm_count, cudaStream_t s);

// Process-wide settings of the bounded waits (pkv_set_wait_limit_ns; 0 = the
// default bound) and the test hook that makes the first CTA of the decode
// partial pass leave its first pipeline stage unfilled
// (pkv_set_debug_skip_fill), read by every launch; and the number of the next
// launch with bounded waits (distinct, nonzero; see WaitCtl).
unsigned long long wait_limit_ns();
int debug_skip_fill();
int next_launch_epoch();

// Shared-prefix decode, prefix pass (on the prefill kernel): the key tiles of
// the shared prefix are split in *nsplit ranges of *per_split tiles so that
// the pass fills the GPU; launch_prefix_pass writes the prefix states of
// every (split, sequence, q head) to pre_ml [nsplit, batch, hq, 2] and
// pre_acc [nsplit, batch, hq, D] (fp32).  Supported where prefill_supported.
void prefix_plan(const PoolView& pv, int num_q_heads, int batch, int prefix_blocks, int sm_count,
                 int* nsplit, int* per_split);
cudaError_t launch_prefix_pass(const PoolView& pv, int layer, const void* q, int num_q_heads,
                               float scale, const int32_t* bt, int mb, const int32_t* lens,
                               const int32_t* offs, int batch, int prefix_blocks, float* pre_ml,
                               float* pre_acc, int* err, int sm_count, cudaStream_t s);

// Current-device facts for entry points defined outside api.cu: dynamic
// shared memory limit, the sticky error word, the decode grid size and the
// validate flag.  Returns a pkv_status value.
int device_facts(int* smem_optin, int** err_word, int* decode_grid, int* validate);
// Validate-mode helpers of api.cu (pkv_status values).
int clear_error_word(int* err, cudaStream_t s);
int read_and_clear_error_word(int* err, cudaStream_t s);

}  // namespace pkv
