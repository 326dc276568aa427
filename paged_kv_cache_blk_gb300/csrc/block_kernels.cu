// Whole-block moves on the pool:
//   pkv_copy_blocks - block dst[i] <- block src[i] (copy-on-write; mini-runtime
//                     ch.12 §3.1)
//   pkv_swap_out    - listed blocks -> contiguous page-locked host buffers
//   pkv_swap_in     - contiguous host buffers -> listed blocks
//                     (preemption by swapping, "vLLM PagedAttention source
//                     notes" §2.4)
// A block's data in one layer is one contiguous run of bs * row bytes; across
// all layers it is one run of L * bs * row bytes (the pool is
// [N, L, bs, Hkv, D]).  One kernel moves runs: CTA (chunk, i) copies up to
// 64 KB of run i with 16-byte vector accesses, all loads of a batch before
// its stores.  Host buffers are read and written in place by the kernel (on
// GB300 over NVLink-C2C); the host checks accept only page-locked host memory
// that CUDA maps for the device.
#include "common.cuh"
#include "pkv.h"

namespace pkv {
namespace {

constexpr int kRunThreads = 256;
constexpr long long kChunk = 64 * 1024;

// src run i starts at src + (src_ids ? src_ids[i] : i) * src_stride; same for
// dst.  Ids outside [0, id_limit) are skipped and flagged.
__global__ void __launch_bounds__(kRunThreads) copy_runs_kernel(
    const char* __restrict__ src, long long src_stride, const int32_t* __restrict__ src_ids,
    char* __restrict__ dst, long long dst_stride, const int32_t* __restrict__ dst_ids, int n,
    long long run_bytes, long long id_limit, int* err) {
  griddep_wait();
  griddep_launch_dependents();
  const int i = blockIdx.y;
  if (i >= n) return;
  const long long si = src_ids ? src_ids[i] : i;
  const long long di = dst_ids ? dst_ids[i] : i;
  if ((src_ids && (si < 0 || si >= id_limit)) || (dst_ids && (di < 0 || di >= id_limit))) {
    if (blockIdx.x == 0 && threadIdx.x == 0) set_error(err, kErrIndex);
    return;
  }
  const long long lo = (long long)blockIdx.x * kChunk;
  if (lo >= run_bytes) return;
  const long long hi = min(run_bytes, lo + kChunk);
  const char* s = src + si * src_stride;
  char* d = dst + di * dst_stride;
  constexpr int U = 4;
  for (long long base = lo + (long long)threadIdx.x * 16; base < hi;
       base += (long long)kRunThreads * 16 * U) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const long long off = base + (long long)u * kRunThreads * 16;
      if (off < hi) v[u] = *reinterpret_cast<const uint4*>(s + off);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const long long off = base + (long long)u * kRunThreads * 16;
      if (off < hi) *reinterpret_cast<uint4*>(d + off) = v[u];
    }
  }
}

cudaError_t launch_runs(const char* src, long long src_stride, const int32_t* src_ids, char* dst,
                        long long dst_stride, const int32_t* dst_ids, int n, long long run_bytes,
                        long long id_limit, int* err, cudaStream_t s) {
  const long long chunks = (run_bytes + kChunk - 1) / kChunk;
  return launch_kernel(copy_runs_kernel, dim3((unsigned)chunks, (unsigned)n), dim3(kRunThreads), 0,
                       s, true, src, src_stride, src_ids, dst, dst_stride, dst_ids, n, run_bytes,
                       id_limit, err);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Geometry of a block move: base offset, run length and block stride.
struct Runs {
  long long base, run, stride;
};

int pool_runs(const pkv_pool* p, int32_t layer, Runs* r) {
  PoolView v;
  const int st = pool_view(p, true, &v);  // geometry, tensors, row bytes of any dtype
  if (st != PKV_OK) return st;
  if (layer < -1 || layer >= p->num_layers) return PKV_ERR_INVALID_ARG;
  const long long layer_run = (long long)p->block_size * v.row_bytes;
  r->stride = layer_run * p->num_layers;
  r->base = layer < 0 ? 0 : layer * layer_run;
  r->run = layer < 0 ? r->stride : layer_run;
  return PKV_OK;
}

// Page-locked host memory the device can address (cudaHostAlloc, or
// cudaHostRegister'd), `bytes` long from p.
bool device_reachable_host(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeHost && a.devicePointer == p;
}

pkv_status finish(cudaError_t e, int* err, int validate, cudaStream_t s) {
  if (e != cudaSuccess) {
    cudaGetLastError();
    return PKV_ERR_CUDA;
  }
  return validate ? static_cast<pkv_status>(read_and_clear_error_word(err, s)) : PKV_OK;
}

}  // namespace
}  // namespace pkv

extern "C" pkv_status pkv_copy_blocks(const pkv_pool* pool, int32_t layer,
                                      const int32_t* src_blocks, const int32_t* dst_blocks,
                                      int32_t num_pairs, cudaStream_t stream) {
  if (!pool) return PKV_ERR_INVALID_ARG;
  pkv::Runs r;
  pkv_status st = static_cast<pkv_status>(pkv::pool_runs(pool, layer, &r));
  if (st != PKV_OK) return st;
  if (num_pairs < 0) return PKV_ERR_INVALID_ARG;
  if (num_pairs == 0) return PKV_OK;
  if (!src_blocks || !dst_blocks) return PKV_ERR_INVALID_ARG;
  int smem = 0, grid = 0, validate = 0;
  int* err = nullptr;
  if ((st = static_cast<pkv_status>(pkv::device_facts(&smem, &err, &grid, &validate))) != PKV_OK)
    return st;
  if (validate && (st = static_cast<pkv_status>(pkv::clear_error_word(err, stream))) != PKV_OK)
    return st;
  for (int t = 0; t < 2; ++t) {
    char* base = static_cast<char*>(t == 0 ? pool->k_cache : pool->v_cache) + r.base;
    const cudaError_t e = pkv::launch_runs(base, r.stride, src_blocks, base, r.stride, dst_blocks,
                                           num_pairs, r.run, pool->num_blocks, err, stream);
    if (e != cudaSuccess) return pkv::finish(e, err, 0, stream);
  }
  return pkv::finish(cudaSuccess, err, validate, stream);
}

extern "C" pkv_status pkv_swap_out(const pkv_pool* pool, int32_t layer, const int32_t* blocks,
                                   int32_t n, void* host_k, void* host_v, size_t host_bytes,
                                   cudaStream_t stream) {
  if (!pool) return PKV_ERR_INVALID_ARG;
  pkv::Runs r;
  pkv_status st = static_cast<pkv_status>(pkv::pool_runs(pool, layer, &r));
  if (st != PKV_OK) return st;
  if (n < 0) return PKV_ERR_INVALID_ARG;
  if (n == 0) return PKV_OK;
  if (!blocks || !host_k || !host_v || !pkv::aligned16(host_k) || !pkv::aligned16(host_v))
    return PKV_ERR_INVALID_ARG;
  if ((unsigned long long)n * (unsigned long long)r.run > host_bytes) return PKV_ERR_INVALID_ARG;
  if (!pkv::device_reachable_host(host_k) || !pkv::device_reachable_host(host_v))
    return PKV_ERR_INVALID_ARG;
  int smem = 0, grid = 0, validate = 0;
  int* err = nullptr;
  if ((st = static_cast<pkv_status>(pkv::device_facts(&smem, &err, &grid, &validate))) != PKV_OK)
    return st;
  if (validate && (st = static_cast<pkv_status>(pkv::clear_error_word(err, stream))) != PKV_OK)
    return st;
  for (int t = 0; t < 2; ++t) {
    const char* base = static_cast<const char*>(t == 0 ? pool->k_cache : pool->v_cache) + r.base;
    char* host = static_cast<char*>(t == 0 ? host_k : host_v);
    const cudaError_t e = pkv::launch_runs(base, r.stride, blocks, host, r.run, nullptr, n, r.run,
                                           pool->num_blocks, err, stream);
    if (e != cudaSuccess) return pkv::finish(e, err, 0, stream);
  }
  return pkv::finish(cudaSuccess, err, validate, stream);
}

extern "C" pkv_status pkv_swap_in(const pkv_pool* pool, int32_t layer, const int32_t* blocks,
                                  int32_t n, const void* host_k, const void* host_v,
                                  size_t host_bytes, cudaStream_t stream) {
  if (!pool) return PKV_ERR_INVALID_ARG;
  pkv::Runs r;
  pkv_status st = static_cast<pkv_status>(pkv::pool_runs(pool, layer, &r));
  if (st != PKV_OK) return st;
  if (n < 0) return PKV_ERR_INVALID_ARG;
  if (n == 0) return PKV_OK;
  if (!blocks || !host_k || !host_v || !pkv::aligned16(host_k) || !pkv::aligned16(host_v))
    return PKV_ERR_INVALID_ARG;
  if ((unsigned long long)n * (unsigned long long)r.run > host_bytes) return PKV_ERR_INVALID_ARG;
  if (!pkv::device_reachable_host(host_k) || !pkv::device_reachable_host(host_v))
    return PKV_ERR_INVALID_ARG;
  int smem = 0, grid = 0, validate = 0;
  int* err = nullptr;
  if ((st = static_cast<pkv_status>(pkv::device_facts(&smem, &err, &grid, &validate))) != PKV_OK)
    return st;
  if (validate && (st = static_cast<pkv_status>(pkv::clear_error_word(err, stream))) != PKV_OK)
    return st;
  for (int t = 0; t < 2; ++t) {
    char* base = static_cast<char*>(t == 0 ? pool->k_cache : pool->v_cache) + r.base;
    const char* host = static_cast<const char*>(t == 0 ? host_k : host_v);
    const cudaError_t e = pkv::launch_runs(host, r.run, nullptr, base, r.stride, blocks, n, r.run,
                                           pool->num_blocks, err, stream);
    if (e != cudaSuccess) return pkv::finish(e, err, 0, stream);
  }
  return pkv::finish(cudaSuccess, err, validate, stream);
}
