// C ABI of libpkv: argument checks, device bookkeeping, validate mode and
// dispatch to the kernels.  See include/pkv.h for the contract of each call.
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "pkv.h"

namespace {

// Per device context: [0] the sticky error word, into which kernels OR
// pkv::kErr* bits through the pointer obtained for the current device;
// [1] the abort word, holding the number of the last launch whose bounded
// wait gave up (see pkv::WaitCtl).  Both are cleared together.
__device__ int g_pkv_error_word[2];

std::atomic<int> g_validate{0};
std::atomic<int> g_decode_ctas{0};
std::atomic<cudaEvent_t> g_ev_start{nullptr};
std::atomic<cudaEvent_t> g_ev_stop{nullptr};
std::atomic<unsigned long long> g_wait_ns{0};
std::atomic<int> g_skip_fill{0};
std::atomic<unsigned> g_epoch{0};

constexpr int kMaxDevices = 64;

struct DevInfo {
  std::atomic<bool> ready{false};
  int sm_count = 0;
  int smem_optin = 0;
  int* err = nullptr;
};

DevInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

pkv_status current_device(DevInfo** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return PKV_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return PKV_ERR_UNSUPPORTED;
  DevInfo& d = g_dev[dev];
  if (!d.ready.load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(g_dev_mu);
    if (!d.ready.load(std::memory_order_relaxed)) {
      int sms = 0, optin = 0;
      void* err = nullptr;
      if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
              cudaSuccess ||
          cudaGetSymbolAddress(&err, g_pkv_error_word) != cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_CUDA;
      }
      d.sm_count = sms;
      d.smem_optin = optin;
      d.err = static_cast<int*>(err);
      d.ready.store(true, std::memory_order_release);
    }
  }
  *out = &d;
  return PKV_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

int elem_size(int32_t dtype) {
  return dtype == PKV_F32 ? 4 : dtype == PKV_BF16 ? 2 : dtype == PKV_I8 ? 1 : 0;
}

// Geometry checks shared by every call; `need_ptrs` also checks the tensors.
pkv_status check_pool(const pkv_pool* p, bool need_ptrs, pkv::PoolView* v) {
  if (!p) return PKV_ERR_INVALID_ARG;
  const int es = elem_size(p->dtype);
  if (es == 0) return PKV_ERR_UNSUPPORTED;
  if (p->num_blocks <= 0 || p->num_layers <= 0 || p->num_kv_heads <= 0 || p->head_dim <= 0)
    return PKV_ERR_INVALID_ARG;
  if (!pow2(p->block_size) || p->block_size > 1024) return PKV_ERR_INVALID_ARG;
  const long long elems = (long long)p->num_kv_heads * p->head_dim;
  if (elems > (1ll << 28)) return PKV_ERR_UNSUPPORTED;
  const bool quant = p->dtype == PKV_I8;
  // int8 rows: codes, then one fp32 scale per kv head padded to 16 bytes
  const long long row =
      quant ? elems + (4ll * p->num_kv_heads + 15) / 16 * 16 : elems * es;
  if ((elems * es) % 16 != 0) return PKV_ERR_UNSUPPORTED;
  if (need_ptrs) {
    if (!p->k_cache || !p->v_cache) return PKV_ERR_INVALID_ARG;
    if (!aligned16(p->k_cache) || !aligned16(p->v_cache)) return PKV_ERR_INVALID_ARG;
  }
  v->k = static_cast<const char*>(p->k_cache);
  v->v = static_cast<const char*>(p->v_cache);
  v->k_mut = static_cast<char*>(p->k_cache);
  v->v_mut = static_cast<char*>(p->v_cache);
  v->num_blocks = p->num_blocks;
  v->num_layers = p->num_layers;
  v->block_size = p->block_size;
  v->num_kv_heads = p->num_kv_heads;
  v->head_dim = p->head_dim;
  v->elem_size = es;
  v->row_bytes = (int)row;
  v->quant = quant ? 1 : 0;
  v->io_size = quant ? 2 : es;
  v->scale_off = quant ? (int)elems : 0;
  return PKV_OK;
}

pkv_status map_bits(int bits) {
  if (bits & pkv::kErrTimeout) return PKV_ERR_TIMEOUT;
  if (bits & pkv::kErrIndex) return PKV_ERR_INDEX;
  if (bits & pkv::kErrCapacity) return PKV_ERR_CAPACITY;
  return PKV_OK;
}

// Wait for `s`, read the error word and reset it.
pkv_status read_and_clear(int* err, cudaStream_t s) {
  int h = 0;
  if (cudaMemcpyAsync(&h, err, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return PKV_ERR_CUDA;
  }
  if (h != 0) {
    if (cudaMemsetAsync(err, 0, 2 * sizeof(int), s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
      cudaGetLastError();
      return PKV_ERR_CUDA;
    }
  }
  return map_bits(h);
}

pkv_status clear_word(int* err, cudaStream_t s) {
  if (cudaMemsetAsync(err, 0, 2 * sizeof(int), s) != cudaSuccess) {
    cudaGetLastError();
    return PKV_ERR_CUDA;
  }
  return PKV_OK;
}

pkv_status launched(cudaError_t e) {
  if (e != cudaSuccess) {
    cudaGetLastError();
    return PKV_ERR_CUDA;
  }
  return PKV_OK;
}

int decode_grid(const DevInfo& d) {
  const int forced = g_decode_ctas.load();
  return forced > 0 ? forced : d.sm_count;
}

}  // namespace

namespace pkv {

int pool_view(const pkv_pool* p, bool need_ptrs, PoolView* v) {
  return check_pool(p, need_ptrs, v);
}

int device_facts(int* smem_optin, int** err_word, int* grid, int* validate) {
  DevInfo* d;
  const pkv_status st = current_device(&d);
  if (st != PKV_OK) return st;
  *smem_optin = d->smem_optin;
  *err_word = d->err;
  *grid = decode_grid(*d);
  *validate = g_validate.load();
  return PKV_OK;
}

unsigned long long wait_limit_ns() { return g_wait_ns.load(); }

int debug_skip_fill() { return g_skip_fill.load(); }

int next_launch_epoch() {
  unsigned e = g_epoch.fetch_add(1) + 1;
  while ((e & 0x7fffffffu) == 0) e = g_epoch.fetch_add(1) + 1;
  return (int)(e & 0x7fffffffu);
}

int clear_error_word(int* err, cudaStream_t s) { return clear_word(err, s); }

int read_and_clear_error_word(int* err, cudaStream_t s) { return read_and_clear(err, s); }

}  // namespace pkv

extern "C" {

pkv_status pkv_build_slot_mapping(const pkv_pool* pool, const int32_t* block_tables,
                                  int32_t max_blocks_per_seq, const int32_t* offsets,
                                  int32_t batch, const int32_t* token_seq,
                                  const int32_t* token_pos, int64_t num_tokens,
                                  int64_t* slot_mapping, cudaStream_t stream) {
  pkv::PoolView v;
  pkv_status st = check_pool(pool, false, &v);
  if (st != PKV_OK) return st;
  if (num_tokens < 0 || batch < 0) return PKV_ERR_INVALID_ARG;
  if (num_tokens == 0) return PKV_OK;
  if (!token_seq || !token_pos || !slot_mapping) return PKV_ERR_INVALID_ARG;
  if (!aligned(slot_mapping, 8) || !aligned(token_seq, 4) || !aligned(token_pos, 4))
    return PKV_ERR_INVALID_ARG;
  if (batch > 0 && (!block_tables || max_blocks_per_seq <= 0)) return PKV_ERR_INVALID_ARG;
  DevInfo* d;
  if ((st = current_device(&d)) != PKV_OK) return st;
  const bool validate = g_validate.load() != 0;
  if (validate) {
    if ((st = clear_word(d->err, stream)) != PKV_OK) return st;
    if ((st = launched(pkv::launch_validate_tokens(v, block_tables, max_blocks_per_seq, offsets,
                                                   batch, token_seq, token_pos, num_tokens,
                                                   d->err, stream))) != PKV_OK)
      return st;
    if ((st = read_and_clear(d->err, stream)) != PKV_OK) return st;
  }
  if ((st = launched(pkv::launch_slot_mapping(v, block_tables, max_blocks_per_seq, offsets, batch,
                                              token_seq, token_pos, num_tokens, slot_mapping,
                                              d->err, stream))) != PKV_OK)
    return st;
  return validate ? read_and_clear(d->err, stream) : PKV_OK;
}

pkv_status pkv_write_slots(const pkv_pool* pool, int32_t layer, const void* k_new,
                           const void* v_new, const int64_t* slot_mapping, int64_t num_tokens,
                           cudaStream_t stream) {
  pkv::PoolView v;
  pkv_status st = check_pool(pool, true, &v);
  if (st != PKV_OK) return st;
  if (layer < 0 || layer >= pool->num_layers || num_tokens < 0) return PKV_ERR_INVALID_ARG;
  if (num_tokens == 0) return PKV_OK;
  if (v.quant && v.head_dim != 32 && v.head_dim != 64 && v.head_dim != 128 && v.head_dim != 256)
    return PKV_ERR_UNSUPPORTED;
  if (!k_new || !v_new || !slot_mapping) return PKV_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned(slot_mapping, 8))
    return PKV_ERR_INVALID_ARG;
  DevInfo* d;
  if ((st = current_device(&d)) != PKV_OK) return st;
  const bool validate = g_validate.load() != 0;
  if (validate) {
    if ((st = clear_word(d->err, stream)) != PKV_OK) return st;
    if ((st = launched(pkv::launch_validate_slots(v, slot_mapping, num_tokens, d->err, stream))) !=
        PKV_OK)
      return st;
    if ((st = read_and_clear(d->err, stream)) != PKV_OK) return st;
  }
  if ((st = launched(pkv::launch_write_slots(v, layer, k_new, v_new, slot_mapping, num_tokens,
                                             d->err, d->sm_count, stream))) != PKV_OK)
    return st;
  return validate ? read_and_clear(d->err, stream) : PKV_OK;
}

pkv_status pkv_append_tokens(const pkv_pool* pool, int32_t layer, const int32_t* block_tables,
                             int32_t max_blocks_per_seq, const int32_t* offsets, int32_t batch,
                             const int32_t* token_seq, const int32_t* token_pos,
                             int64_t num_tokens, const void* k_new, const void* v_new,
                             int64_t* slot_mapping, cudaStream_t stream) {
  pkv::PoolView v;
  pkv_status st = check_pool(pool, true, &v);
  if (st != PKV_OK) return st;
  if (layer < 0 || layer >= pool->num_layers || num_tokens < 0 || batch < 0)
    return PKV_ERR_INVALID_ARG;
  if (v.quant && v.head_dim != 32 && v.head_dim != 64 && v.head_dim != 128 && v.head_dim != 256)
    return PKV_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PKV_OK;
  if (!token_seq || !token_pos || !k_new || !v_new) return PKV_ERR_INVALID_ARG;
  if (!aligned(token_seq, 4) || !aligned(token_pos, 4) || !aligned16(k_new) || !aligned16(v_new))
    return PKV_ERR_INVALID_ARG;
  if (slot_mapping && !aligned(slot_mapping, 8)) return PKV_ERR_INVALID_ARG;
  if (batch > 0 && (!block_tables || max_blocks_per_seq <= 0)) return PKV_ERR_INVALID_ARG;
  DevInfo* d;
  if ((st = current_device(&d)) != PKV_OK) return st;
  const bool validate = g_validate.load() != 0;
  if (validate) {
    if ((st = clear_word(d->err, stream)) != PKV_OK) return st;
    if ((st = launched(pkv::launch_validate_tokens(v, block_tables, max_blocks_per_seq, offsets,
                                                   batch, token_seq, token_pos, num_tokens,
                                                   d->err, stream))) != PKV_OK)
      return st;
    if ((st = read_and_clear(d->err, stream)) != PKV_OK) return st;
  }
  if ((st = launched(pkv::launch_append(v, layer, block_tables, max_blocks_per_seq, offsets,
                                        batch, token_seq, token_pos, num_tokens, k_new, v_new,
                                        slot_mapping, d->err, stream))) != PKV_OK)
    return st;
  return validate ? read_and_clear(d->err, stream) : PKV_OK;
}

pkv_status pkv_gather(const pkv_pool* pool, int32_t layer, const int32_t* block_tables,
                      int32_t max_blocks_per_seq, const int32_t* seq_lens,
                      const int32_t* offsets, int32_t batch, const int64_t* cu_seqlens,
                      int64_t total_tokens, void* k_out, void* v_out, cudaStream_t stream) {
  pkv::PoolView v;
  pkv_status st = check_pool(pool, true, &v);
  if (st != PKV_OK) return st;
  if (layer < 0 || layer >= pool->num_layers || batch < 0 || total_tokens < 0)
    return PKV_ERR_INVALID_ARG;
  if (batch == 0) return total_tokens == 0 ? PKV_OK : PKV_ERR_INVALID_ARG;
  if (!block_tables || max_blocks_per_seq <= 0 || !seq_lens || !cu_seqlens)
    return PKV_ERR_INVALID_ARG;
  if (!aligned(cu_seqlens, 8)) return PKV_ERR_INVALID_ARG;
  if (total_tokens > 0) {
    if (!k_out || !v_out || !aligned16(k_out) || !aligned16(v_out)) return PKV_ERR_INVALID_ARG;
  }
  DevInfo* d;
  if ((st = current_device(&d)) != PKV_OK) return st;
  const bool validate = g_validate.load() != 0;
  if (validate) {
    if ((st = clear_word(d->err, stream)) != PKV_OK) return st;
    if ((st = launched(pkv::launch_validate_tables(v, block_tables, max_blocks_per_seq, seq_lens,
                                                   offsets, batch, cu_seqlens, total_tokens,
                                                   d->err, stream))) != PKV_OK)
      return st;
    if ((st = read_and_clear(d->err, stream)) != PKV_OK) return st;
  }
  if ((st = launched(pkv::launch_gather(v, layer, block_tables, max_blocks_per_seq, offsets, batch,
                                        cu_seqlens, total_tokens, k_out, v_out, d->err,
                                        stream))) != PKV_OK)
    return st;
  return validate ? read_and_clear(d->err, stream) : PKV_OK;
}

size_t pkv_decode_workspace_size(int32_t batch, int32_t num_q_heads, int32_t head_dim) {
  if (batch < 0 || num_q_heads <= 0 || head_dim <= 0) return 0;
  DevInfo* d;
  if (current_device(&d) != PKV_OK) return 0;
  return pkv::decode_workspace_bytes(batch, num_q_heads, head_dim, decode_grid(*d));
}

// Decode attention, and with new K/V rows (k_new != nullptr) the fused
// decode step that first stores them at each sequence's last position.
static pkv_status decode_call(const pkv_pool* pool, int32_t layer, const void* q,
                              int32_t num_q_heads, float scale, const int32_t* block_tables,
                              int32_t max_blocks_per_seq, const int32_t* seq_lens,
                              const int32_t* offsets, int32_t batch, const void* k_new,
                              const void* v_new, bool step, void* out, void* workspace,
                              size_t workspace_bytes, cudaStream_t stream) {
  pkv::PoolView v;
  pkv_status st = check_pool(pool, true, &v);
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
  if (step && (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)))
    return PKV_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace)) return PKV_ERR_WORKSPACE;
  DevInfo* d;
  if ((st = current_device(&d)) != PKV_OK) return st;
  const int grid = decode_grid(*d);
  if (workspace_bytes < pkv::decode_workspace_bytes(batch, num_q_heads, v.head_dim, grid))
    return PKV_ERR_WORKSPACE;
  const bool validate = g_validate.load() != 0;
  if (validate) {
    if ((st = clear_word(d->err, stream)) != PKV_OK) return st;
    if ((st = launched(pkv::launch_validate_tables(v, block_tables, max_blocks_per_seq, seq_lens,
                                                   offsets, batch, nullptr, 0, d->err,
                                                   stream))) != PKV_OK)
      return st;
    if ((st = read_and_clear(d->err, stream)) != PKV_OK) return st;
  }
  const size_t row_elems = (size_t)num_q_heads * v.head_dim;
  cudaEvent_t ev_start = g_ev_start.load(), ev_stop = g_ev_stop.load();
  if (!ev_start || !ev_stop) ev_start = ev_stop = nullptr;
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
    a.workspace = workspace;
    a.grid = grid;
    a.err = d->err;
    a.smem_optin = d->smem_optin;
    a.ev_start = b0 == 0 ? ev_start : nullptr;
    a.ev_stop = b0 + nb >= batch ? ev_stop : nullptr;
    if (step) {
      const size_t in_row = (size_t)v.num_kv_heads * v.head_dim * v.io_size;
      a.k_new = static_cast<const char*>(k_new) + (size_t)b0 * in_row;
      a.v_new = static_cast<const char*>(v_new) + (size_t)b0 * in_row;
    }
    const cudaError_t e = pkv::launch_decode(a, stream);
    if (e == cudaErrorInvalidConfiguration) return PKV_ERR_UNSUPPORTED;
    if ((st = launched(e)) != PKV_OK) return st;
  }
  return validate ? read_and_clear(d->err, stream) : PKV_OK;
}

pkv_status pkv_decode_attention(const pkv_pool* pool, int32_t layer, const void* q,
                                int32_t num_q_heads, float scale, const int32_t* block_tables,
                                int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                const int32_t* offsets, int32_t batch, void* out, void* workspace,
                                size_t workspace_bytes, cudaStream_t stream) {
  return decode_call(pool, layer, q, num_q_heads, scale, block_tables, max_blocks_per_seq,
                     seq_lens, offsets, batch, nullptr, nullptr, false, out, workspace,
                     workspace_bytes, stream);
}

pkv_status pkv_decode_step(const pkv_pool* pool, int32_t layer, const void* q,
                           int32_t num_q_heads, float scale, const int32_t* block_tables,
                           int32_t max_blocks_per_seq, const int32_t* seq_lens,
                           const int32_t* offsets, int32_t batch, const void* k_new,
                           const void* v_new, void* out, void* workspace, size_t workspace_bytes,
                           cudaStream_t stream) {
  return decode_call(pool, layer, q, num_q_heads, scale, block_tables, max_blocks_per_seq,
                     seq_lens, offsets, batch, k_new, v_new, true, out, workspace,
                     workspace_bytes, stream);
}

// Shared-prefix decode: which path a call takes, and the workspace carve of
// the two-pass path ([decode workspace][prefix m, l][prefix acc]).
struct PrefixPlan {
  bool two_pass;  // false: the plain decode path computes the same result
  int nsplit, per_split;
  size_t decode_ws, ml_off, acc_off, total;
};

static PrefixPlan plan_prefix(const pkv::PoolView& v, int32_t batch, int32_t num_q_heads,
                              int32_t prefix_blocks, const DevInfo& d) {
  PrefixPlan pl{};
  const int grid = decode_grid(d);
  pl.decode_ws = pkv::decode_workspace_bytes(batch, num_q_heads, v.head_dim, grid);
  pl.total = pl.decode_ws;
  pl.two_pass = prefix_blocks > 0 && batch > 0 && batch <= pkv::kDecodeMaxBatch &&
                pkv::prefill_supported(v, num_q_heads) == 0 &&
                pkv::decode_supported(v, num_q_heads) == 0;
  if (!pl.two_pass) return pl;
  pkv::prefix_plan(v, num_q_heads, batch, prefix_blocks, d.sm_count, &pl.nsplit, &pl.per_split);
  const size_t rows = (size_t)pl.nsplit * batch * num_q_heads;
  pl.ml_off = (pl.decode_ws + 255) / 256 * 256;
  pl.acc_off = pl.ml_off + (rows * 2 * 4 + 255) / 256 * 256;
  pl.total = pl.acc_off + rows * v.head_dim * 4;
  return pl;
}

size_t pkv_decode_shared_prefix_workspace_size(const pkv_pool* pool, int32_t batch,
                                               int32_t num_q_heads, int32_t num_prefix_blocks) {
  pkv::PoolView v;
  if (check_pool(pool, false, &v) != PKV_OK) return 0;
  if (batch < 0 || num_q_heads <= 0 || num_prefix_blocks < 0) return 0;
  if (num_q_heads % pool->num_kv_heads != 0) return 0;
  DevInfo* d;
  if (current_device(&d) != PKV_OK) return 0;
  return plan_prefix(v, batch, num_q_heads, num_prefix_blocks, *d).total;
}

pkv_status pkv_decode_attention_shared_prefix(const pkv_pool* pool, int32_t layer, const void* q,
                                              int32_t num_q_heads, float scale,
                                              const int32_t* block_tables,
                                              int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                              const int32_t* offsets, int32_t batch,
                                              int32_t num_prefix_blocks, void* out,
                                              void* workspace, size_t workspace_bytes,
                                              cudaStream_t stream) {
  pkv::PoolView v;
  pkv_status st = check_pool(pool, true, &v);
  if (st != PKV_OK) return st;
  if (num_prefix_blocks < 0 || (batch > 0 && num_prefix_blocks > max_blocks_per_seq))
    return PKV_ERR_INVALID_ARG;
  if (layer < 0 || layer >= pool->num_layers || batch < 0 || num_q_heads <= 0)
    return PKV_ERR_INVALID_ARG;
  if (num_q_heads % pool->num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return PKV_ERR_INVALID_ARG;
  if (pkv::decode_supported(v, num_q_heads) != 0) return PKV_ERR_UNSUPPORTED;
  if (batch == 0) return PKV_OK;
  DevInfo* d;
  if ((st = current_device(&d)) != PKV_OK) return st;
  const PrefixPlan pl = plan_prefix(v, batch, num_q_heads, num_prefix_blocks, *d);
  if (!pl.two_pass)
    return decode_call(pool, layer, q, num_q_heads, scale, block_tables, max_blocks_per_seq,
                       seq_lens, offsets, batch, nullptr, nullptr, false, out, workspace,
                       workspace_bytes, stream);
  if (!q || !out || !block_tables || !seq_lens || max_blocks_per_seq <= 0)
    return PKV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(out)) return PKV_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace)) return PKV_ERR_WORKSPACE;
  if (workspace_bytes < pl.total) return PKV_ERR_WORKSPACE;
  const bool validate = g_validate.load() != 0;
  if (validate) {
    if ((st = clear_word(d->err, stream)) != PKV_OK) return st;
    if ((st = launched(pkv::launch_validate_tables(v, block_tables, max_blocks_per_seq, seq_lens,
                                                   offsets, batch, nullptr, 0, d->err,
                                                   stream))) != PKV_OK)
      return st;
    if ((st = launched(pkv::launch_validate_prefix(v, block_tables, max_blocks_per_seq, seq_lens,
                                                   offsets, batch, num_prefix_blocks, d->err,
                                                   stream))) != PKV_OK)
      return st;
    if ((st = read_and_clear(d->err, stream)) != PKV_OK) return st;
  }
  char* ws = static_cast<char*>(workspace);
  float* pre_ml = reinterpret_cast<float*>(ws + pl.ml_off);
  float* pre_acc = reinterpret_cast<float*>(ws + pl.acc_off);
  pkv::DecodeLaunch a;
  a.pool = v;
  a.layer = layer;
  a.q = q;
  a.out = out;
  a.num_q_heads = num_q_heads;
  a.scale = scale;
  a.bt = block_tables;
  a.mb = max_blocks_per_seq;
  a.lens = seq_lens;
  a.offs = offsets;
  a.batch = batch;
  a.workspace = workspace;
  a.grid = decode_grid(*d);
  a.err = d->err;
  a.smem_optin = d->smem_optin;
  a.prefix_blocks = num_prefix_blocks;
  cudaEvent_t ev_start = g_ev_start.load(), ev_stop = g_ev_stop.load();
  if (ev_start && ev_stop) {
    a.ev_start = ev_start;
    a.ev_stop = ev_stop;
  }
  // the suffix pass first: the prefix states written after it stay in L2
  // for the combine
  cudaError_t e = pkv::launch_decode(a, stream);
  if (e == cudaErrorInvalidConfiguration) return PKV_ERR_UNSUPPORTED;
  if ((st = launched(e)) != PKV_OK) return st;
  if ((st = launched(pkv::launch_prefix_pass(v, layer, q, num_q_heads, scale, block_tables,
                                             max_blocks_per_seq, seq_lens, offsets, batch,
                                             num_prefix_blocks, pre_ml, pre_acc, d->err,
                                             d->sm_count, stream))) != PKV_OK)
    return st;
  if ((st = launched(pkv::launch_decode_combine_prefix(a, pre_ml, pre_acc, pl.nsplit, stream))) !=
      PKV_OK)
    return st;
  return validate ? read_and_clear(d->err, stream) : PKV_OK;
}

pkv_status pkv_prefill_attention(const pkv_pool* pool, int32_t layer, const void* q,
                                 int32_t num_q_heads, float scale, const int32_t* block_tables,
                                 int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                 const int32_t* offsets, const int64_t* cu_q, int32_t batch,
                                 int64_t total_q, int32_t max_q_len, void* out,
                                 cudaStream_t stream) {
  pkv::PoolView v;
  pkv_status st = check_pool(pool, true, &v);
  if (st != PKV_OK) return st;
  if (layer < 0 || layer >= pool->num_layers || batch < 0 || num_q_heads <= 0 || total_q < 0 ||
      max_q_len < 0)
    return PKV_ERR_INVALID_ARG;
  if (num_q_heads % pool->num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return PKV_ERR_INVALID_ARG;
  if (pkv::prefill_supported(v, num_q_heads) != 0) return PKV_ERR_UNSUPPORTED;
  if (batch == 0 || total_q == 0 || max_q_len == 0) return PKV_OK;
  if (batch > 65535 || total_q > INT32_MAX) return PKV_ERR_UNSUPPORTED;
  if (!q || !out || !block_tables || !seq_lens || !cu_q || max_blocks_per_seq <= 0)
    return PKV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(out) || !aligned(cu_q, 8)) return PKV_ERR_INVALID_ARG;
  DevInfo* d;
  if ((st = current_device(&d)) != PKV_OK) return st;
  const bool validate = g_validate.load() != 0;
  if (validate) {
    if ((st = clear_word(d->err, stream)) != PKV_OK) return st;
    if ((st = launched(pkv::launch_validate_tables(v, block_tables, max_blocks_per_seq, seq_lens,
                                                   offsets, batch, nullptr, 0, d->err,
                                                   stream))) != PKV_OK)
      return st;
    if ((st = read_and_clear(d->err, stream)) != PKV_OK) return st;
  }
  if ((st = launched(pkv::launch_prefill(v, layer, q, num_q_heads, scale, block_tables,
                                         max_blocks_per_seq, seq_lens, offsets, cu_q, batch,
                                         total_q, max_q_len, out, d->err, d->sm_count, stream))) != PKV_OK)
    return st;
  return validate ? read_and_clear(d->err, stream) : PKV_OK;
}

pkv_status pkv_set_decode_ctas(int32_t num_ctas) {
  if (num_ctas < 0 || num_ctas > 65536) return PKV_ERR_INVALID_ARG;
  g_decode_ctas.store(num_ctas);
  return PKV_OK;
}

pkv_status pkv_set_decode_events(cudaEvent_t start, cudaEvent_t stop) {
  g_ev_start.store(start);
  g_ev_stop.store(stop);
  return PKV_OK;
}

pkv_status pkv_set_wait_limit_ns(uint64_t ns) {
  if (ns != 0 && (ns < 1000ull || ns > 60000000000ull)) return PKV_ERR_INVALID_ARG;
  g_wait_ns.store(ns);
  return PKV_OK;
}

uint64_t pkv_get_wait_limit_ns(void) {
  const unsigned long long ns = g_wait_ns.load();
  return ns ? ns : 4000000000ull;
}

pkv_status pkv_set_debug_skip_fill(int32_t mode) {
  if (mode < 0 || mode > 2) return PKV_ERR_INVALID_ARG;
  g_skip_fill.store(mode);
  return PKV_OK;
}

pkv_status pkv_set_validate(int32_t on) {
  g_validate.store(on ? 1 : 0);
  return PKV_OK;
}

int32_t pkv_get_validate(void) { return g_validate.load(); }

pkv_status pkv_device_error(pkv_status* status, int32_t clear) {
  if (!status) return PKV_ERR_INVALID_ARG;
  DevInfo* d;
  pkv_status st = current_device(&d);
  if (st != PKV_OK) return st;
  int h = 0;
  if (cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpy(&h, d->err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return PKV_ERR_CUDA;
  }
  if (clear && cudaMemset(d->err, 0, 2 * sizeof(int)) != cudaSuccess) {
    cudaGetLastError();
    return PKV_ERR_CUDA;
  }
  *status = map_bits(h);
  return PKV_OK;
}

const char* pkv_status_string(pkv_status status) {
  switch (status) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARG: return "invalid argument";
    case PKV_ERR_CAPACITY: return "sequence exceeds its block table capacity or bad offset";
    case PKV_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case PKV_ERR_WORKSPACE: return "workspace missing or too small";
    case PKV_ERR_INDEX: return "slot or block id out of range";
    case PKV_ERR_CUDA: return "CUDA error";
    case PKV_ERR_TIMEOUT: return "device wait timed out";
    case PKV_ERR_NO_BLOCKS: return "too few free blocks (nothing changed)";
  }
  return "unknown status";
}

int32_t pkv_version(void) { return 100; }

}  // extern "C"
