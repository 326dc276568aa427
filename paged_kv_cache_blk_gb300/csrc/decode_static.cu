// Allocation-free entry point for paged decode attention.
//
// Some callers cannot allocate device memory where they run decode attention:
// serving processes whose memory manager reserves the GPU's memory up front
// and hands out nothing on the hot path, plugin runtimes whose execute step
// must not allocate, and plain C programs that link only this library and
// have no device allocator of their own for scratch.  For them,
// pkv_decode_attention_static keeps the split-K scratch of the decode pass in
// a fixed array in device global memory that this file defines, so the caller
// passes only inputs and outputs.  It runs the same kernels as
// pkv_decode_attention and allocates nothing (no cudaMalloc, no cudaFree, no
// allocating library routine).
//
// The array (PKV_DECODE_STATIC_SCRATCH_BYTES) exists once per GPU that loads
// the library and lives until the process exits.  In host code its name is a
// host-side stand-in, not a device address, so the device address is looked
// up here with cudaGetSymbolAddress, once per device with that device current;
// the first call on a device does that lookup (make it before any stream
// capture).  Every call on a device shares the array and finds the previous
// call's contents in it; the decode pass writes every scratch word before it
// reads it, so nothing needs clearing.  Calls whose kernels overlap on the GPU
// race on the array; calls ordered on one stream are safe.
#include <atomic>
#include <cmath>
#include <mutex>

#include "common.cuh"
#include "pkv.h"

namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[PKV_DECODE_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

struct ScratchAddr {
  std::atomic<bool> ready{false};
  void* ptr = nullptr;
};

ScratchAddr g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of g_decode_scratch on the current device.
pkv_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return PKV_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return PKV_ERR_UNSUPPORTED;
  ScratchAddr& a = g_scratch_addr[dev];
  if (!a.ready.load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!a.ready.load(std::memory_order_relaxed)) {
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess || ptr == nullptr) {
        cudaGetLastError();
        return PKV_ERR_CUDA;
      }
      a.ptr = ptr;
      a.ready.store(true, std::memory_order_release);
    }
  }
  *out = a.ptr;
  return PKV_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" pkv_status pkv_decode_attention_static(const pkv_pool* pool, int32_t layer,
                                                  const void* q, int32_t num_q_heads, float scale,
                                                  const int32_t* block_tables,
                                                  int32_t max_blocks_per_seq,
                                                  const int32_t* seq_lens, const int32_t* offsets,
                                                  int32_t batch, void* out, cudaStream_t stream) {
  // ---- host-visible argument checks (same rules as pkv_decode_attention) ----
  pkv::PoolView v;
  pkv_status st = static_cast<pkv_status>(pkv::pool_view(pool, true, &v));
  if (st != PKV_OK) return st;
  if (layer < 0 || layer >= pool->num_layers || batch < 0 || num_q_heads <= 0)
    return PKV_ERR_INVALID_ARG;
  if (num_q_heads % pool->num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return PKV_ERR_INVALID_ARG;
  if (pkv::decode_supported(v, num_q_heads) != 0) return PKV_ERR_UNSUPPORTED;
  if (batch == 0) return PKV_OK;
  if (!q || !out || !block_tables || !seq_lens || max_blocks_per_seq <= 0)
    return PKV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(out)) return PKV_ERR_INVALID_ARG;

  int smem_optin = 0, grid = 0, validate = 0;
  int* err = nullptr;
  st = static_cast<pkv_status>(pkv::device_facts(&smem_optin, &err, &grid, &validate));
  if (st != PKV_OK) return st;
  // the fixed array bounds the shape: refuse what does not fit
  if (pkv::decode_workspace_bytes(batch, num_q_heads, v.head_dim, grid) >
      PKV_DECODE_STATIC_SCRATCH_BYTES)
    return PKV_ERR_WORKSPACE;
  void* scratch = nullptr;
  if ((st = scratch_address(&scratch)) != PKV_OK) return st;

  if (validate) {
    if ((st = static_cast<pkv_status>(pkv::clear_error_word(err, stream))) != PKV_OK) return st;
    if (pkv::launch_validate_tables(v, block_tables, max_blocks_per_seq, seq_lens, offsets, batch,
                                    nullptr, 0, err, stream) != cudaSuccess) {
      cudaGetLastError();
      return PKV_ERR_CUDA;
    }
    if ((st = static_cast<pkv_status>(pkv::read_and_clear_error_word(err, stream))) != PKV_OK)
      return st;
  }
  const size_t row_elems = (size_t)num_q_heads * v.head_dim;
  for (int b0 = 0; b0 < batch; b0 += pkv::kDecodeMaxBatch) {
    const int nb = batch - b0 < pkv::kDecodeMaxBatch ? batch - b0 : pkv::kDecodeMaxBatch;
    pkv::DecodeLaunch a;
    a.pool = v;
    a.layer = layer;
    a.q = static_cast<const char*>(q) + b0 * row_elems * v.io_size;
    a.out = static_cast<char*>(out) + b0 * row_elems * v.io_size;
    a.num_q_heads = num_q_heads;
    a.scale = scale;
    a.bt = block_tables + (size_t)b0 * max_blocks_per_seq;
    a.mb = max_blocks_per_seq;
    a.lens = seq_lens + b0;
    a.offs = offsets ? offsets + b0 : nullptr;
    a.batch = nb;
    a.workspace = scratch;
    a.grid = grid;
    a.err = err;
    a.smem_optin = smem_optin;
    const cudaError_t e = pkv::launch_decode(a, stream);
    if (e == cudaErrorInvalidConfiguration) return PKV_ERR_UNSUPPORTED;
    if (e != cudaSuccess) {
      cudaGetLastError();
      return PKV_ERR_CUDA;
    }
  }
  return validate ? static_cast<pkv_status>(pkv::read_and_clear_error_word(err, stream)) : PKV_OK;
}
