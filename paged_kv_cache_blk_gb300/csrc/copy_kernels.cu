// Index and copy kernels of the paged KV cache:
//   slot mapping  - logical (sequence, position) -> physical slot
//                   ("vLLM PagedAttention source notes" §2.2 slot_mapping;
//                    mini-runtime ch.12 §2.2 first-block offset)
//   scatter       - slot_mapping write of new K/V rows
//                   ("step14_2 - index_select gather", Relation to step14_1)
//   gather        - block_table read to contiguous [seq_len, Hkv, D]
//                   ("step14_2 - index_select gather", Problem / Solution)
//   validation    - index checks run before the main kernels in validate mode
//
// Scatter and gather are pure copies of whole token rows (Hkv * D elements,
// 16-byte multiple).  One warp moves one token's K row and V row with 16-byte
// vector accesses: 32 lanes cover 512 contiguous bytes per instruction, so
// every access is fully coalesced, and each lane keeps all its loads in
// flight before storing.  Rows are independent, so the grid simply has one
// warp per row; the HBM system sees (rows x 4 x row_bytes) of traffic and no
// re-reads.
#include "common.cuh"
#include "quant.cuh"

namespace pkv {
namespace {

constexpr int kCopyWarps = 8;              // warps per CTA
constexpr int kCopyThreads = kCopyWarps * 32;
constexpr int kMaxVecPerLane = 4;          // vectors per lane kept in flight per tensor

// Copy one K row and one V row (row_vecs 16-byte vectors each) with the
// whole warp: all loads of a chunk are issued before any store.
__device__ __forceinline__ void copy_row_pair(char* dk, const char* sk, char* dv, const char* sv,
                                              int row_vecs, int lane) {
  for (int base = 0; base < row_vecs; base += 32 * kMaxVecPerLane) {
    uint4 a[kMaxVecPerLane], b[kMaxVecPerLane];
#pragma unroll
    for (int u = 0; u < kMaxVecPerLane; ++u) {
      const int v = base + u * 32 + lane;
      if (v < row_vecs) {
        a[u] = ld_stream(sk + 16 * (size_t)v);
        b[u] = ld_stream(sv + 16 * (size_t)v);
      }
    }
#pragma unroll
    for (int u = 0; u < kMaxVecPerLane; ++u) {
      const int v = base + u * 32 + lane;
      if (v < row_vecs) {
        st_global(dk + 16 * (size_t)v, a[u]);
        st_global(dv + 16 * (size_t)v, b[u]);
      }
    }
  }
}

// Byte offset of row j of block `blk` in layer `layer`.
__device__ __forceinline__ long long row_offset(long long blk, int layer, int j, int L, int bs,
                                                int row_bytes) {
  return ((blk * L + layer) * (long long)bs + j) * (long long)row_bytes;
}

// ---------------------------------------------------------------------------
// slot mapping: one thread per token
// ---------------------------------------------------------------------------
// Where the slots of a scatter come from: read from slot_mapping, or (the
// fused append) computed from (sequence, position) pairs through the tables.
struct SlotSrc {
  const int64_t* slots;  // read when not fused
  const int32_t* bt;
  const int32_t* offs;
  const int32_t* tok_seq;
  const int32_t* tok_pos;
  int64_t* slots_out;  // fused: also written here when not null
  int mb, batch;
};

// Slot of token t from its (sequence, position): -1 for padding (negative
// sequence) and for anything out of range (recorded in the error word when
// `report`).
__device__ __forceinline__ int64_t token_slot(const SlotSrc& ss, long long t, long long num_blocks,
                                              int bs, int* err, bool report) {
  const int b = ss.tok_seq[t];
  if (b < 0) return -1;
  if (b >= ss.batch) {
    if (report) set_error(err, kErrIndex);
    return -1;
  }
  const int off = ss.offs ? ss.offs[b] : 0;
  const long long p = (long long)off + ss.tok_pos[t];
  if (off < 0 || off >= bs || ss.tok_pos[t] < 0 || p >= (long long)ss.mb * bs) {
    if (report) set_error(err, kErrCapacity);
    return -1;
  }
  const int blk = ss.bt[(long long)b * ss.mb + p / bs];
  if (blk < 0 || blk >= num_blocks) {
    if (report) set_error(err, kErrIndex);
    return -1;
  }
  return (int64_t)blk * bs + p % bs;
}

__global__ void slot_mapping_kernel(const SlotSrc ss, long long n, long long num_blocks, int bs,
                                    int* err) {
  griddep_wait();
  griddep_launch_dependents();
  for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < n;
       t += (long long)gridDim.x * blockDim.x)
    ss.slots_out[t] = token_slot(ss, t, num_blocks, bs, err, true);
}

// The slot of token t for a scatter: read, or computed (fused append) by
// lane 0 and broadcast to the warp; the warp that `reports` also writes the
// slot out and records errors.
template <bool FUSED>
__device__ __forceinline__ int64_t scatter_slot(const SlotSrc& ss, long long t,
                                                long long num_blocks, int bs, int* err,
                                                bool report, int lane) {
  if constexpr (!FUSED) {
    return ss.slots[t];
  } else {
    int64_t s = 0;
    if (lane == 0) {
      s = token_slot(ss, t, num_blocks, bs, err, report);
      if (report && ss.slots_out) ss.slots_out[t] = s;
    }
    return __shfl_sync(0xffffffffu, s, 0);
  }
}

// ---------------------------------------------------------------------------
// scatter: one warp per token (K row + V row)
// ---------------------------------------------------------------------------
template <bool FUSED>
__global__ void __launch_bounds__(kCopyThreads) write_slots_kernel(
    char* __restrict__ kc, char* __restrict__ vc, const char* __restrict__ k_new,
    const char* __restrict__ v_new, const SlotSrc ss, long long n, long long num_blocks, int L,
    int layer, int bs, int row_bytes, int* err) {
  griddep_wait();
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const long long warps = (long long)gridDim.x * kCopyWarps;
  const int row_vecs = row_bytes >> 4;
  for (long long t = blockIdx.x * (long long)kCopyWarps + (threadIdx.x >> 5); t < n; t += warps) {
    const int64_t s = scatter_slot<FUSED>(ss, t, num_blocks, bs, err, true, lane);
    if (s < 0) {
      if (s != -1 && lane == 0) set_error(err, kErrIndex);
      continue;  // -1 is padding: that row is not written
    }
    if (s >= num_blocks * bs) {
      if (lane == 0) set_error(err, kErrIndex);
      continue;
    }
    const long long dst = row_offset(s / bs, layer, (int)(s % bs), L, bs, row_bytes);
    const long long src = t * (long long)row_bytes;
    copy_row_pair(kc + dst, k_new + src, vc + dst, v_new + src, row_vecs, lane);
  }
}

// ---------------------------------------------------------------------------
// quantising scatter (int8 pools): one warp per (token, kv head), K and V.
// The D bf16 values of the head are spread D/32 per lane; the absmax is a
// warp max over |x| bit patterns (the order of non-negative IEEE numbers),
// scale = absmax / 127 and code = round_half_even(x / scale), both quotients
// IEEE fp32 with subnormals kept (div.rn.f32 without .ftz, whatever the
// fast-math flags), codes clamped to [-127, 127].  A zero absmax stores
// scale 0 and codes 0.  The padding bytes of the row are not written.
// ---------------------------------------------------------------------------
template <int VPL, bool FUSED>
__global__ void __launch_bounds__(kCopyThreads) quant_write_slots_kernel(
    char* __restrict__ kc, char* __restrict__ vc, const __nv_bfloat16* __restrict__ k_new,
    const __nv_bfloat16* __restrict__ v_new, const SlotSrc ss, long long n, long long num_blocks,
    int L, int layer, int bs, int row_bytes, int hkv, int scale_off, int* err) {
  griddep_wait();
  griddep_launch_dependents();
  constexpr int D = 32 * VPL;
  const int lane = threadIdx.x & 31;
  const long long tasks = n * hkv;
  const long long warps = (long long)gridDim.x * kCopyWarps;
  for (long long w = blockIdx.x * (long long)kCopyWarps + (threadIdx.x >> 5); w < tasks;
       w += warps) {
    const long long t = w / hkv;
    const int g = (int)(w - t * hkv);
    const int64_t s = scatter_slot<FUSED>(ss, t, num_blocks, bs, err, g == 0, lane);
    if (s < 0) {
      if (s != -1 && lane == 0 && g == 0) set_error(err, kErrIndex);
      continue;  // -1 is padding: that row is not written
    }
    if (s >= num_blocks * bs) {
      if (lane == 0 && g == 0) set_error(err, kErrIndex);
      continue;
    }
    const long long row = row_offset(s / bs, layer, (int)(s % bs), L, bs, row_bytes);
    const long long src = (t * hkv + g) * D + lane * VPL;
    float xk[VPL], xv[VPL];
    load_bf16<VPL>(k_new + src, xk);
    load_bf16<VPL>(v_new + src, xv);
    int ck[VPL], cv[VPL];
    const float sk = quantise_head<VPL>(xk, ck);
    const float sv = quantise_head<VPL>(xv, cv);
    store_codes<VPL>(kc + row + g * D + lane * VPL, ck);
    store_codes<VPL>(vc + row + g * D + lane * VPL, cv);
    if (lane == 0) {
      *reinterpret_cast<float*>(kc + row + scale_off + 4 * g) = sk;
      *reinterpret_cast<float*>(vc + row + scale_off + 4 * g) = sv;
    }
  }
}

// ---------------------------------------------------------------------------
// gather: one warp per kGatherRows consecutive output rows.  The sequence of
// the first row is found by binary search in the packed layout cu_seqlens
// (small and cache-resident), and the warp walks forward from it, so the
// search is paid once per group.  On the gather_scatter workload 2 rows per
// warp measured best: 3 % faster than 1 and 4 rows, 6 % faster than 8 (with
// more rows per warp, fewer warps share the copy and the last wave is short)
// ---------------------------------------------------------------------------
constexpr int kGatherRows = 2;

__global__ void __launch_bounds__(kCopyThreads) gather_kernel(
    const char* __restrict__ kc, const char* __restrict__ vc, const int32_t* __restrict__ bt,
    int mb, const int32_t* __restrict__ offs, int batch, const int64_t* __restrict__ cu,
    long long total, char* __restrict__ k_out, char* __restrict__ v_out, long long num_blocks,
    int L, int layer, int bs, int row_bytes, int* err) {
  griddep_wait();
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int row_vecs = row_bytes >> 4;
  const long long warps = (long long)gridDim.x * kCopyWarps;
  for (long long r0 = (blockIdx.x * (long long)kCopyWarps + (threadIdx.x >> 5)) * kGatherRows;
       r0 < total; r0 += warps * kGatherRows) {
    // largest b with cu[b] <= r0
    int lo = 0, hi = batch;  // answer in [0, batch)
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (cu[mid] <= r0) lo = mid; else hi = mid;
    }
    int b = lo;
    long long seq_end = cu[b + 1];
    const long long r1 = r0 + kGatherRows < total ? r0 + kGatherRows : total;
    for (long long r = r0; r < r1; ++r) {
      // past the end of sequence b (and any empty ones after it)
      while (r >= seq_end && b + 1 < batch) {
        ++b;
        seq_end = cu[b + 1];
      }
      const long long i = r - cu[b];
      if (i < 0 || r >= seq_end) {  // row not covered by the packed layout
        if (lane == 0) set_error(err, kErrIndex);
        continue;
      }
      const int off = offs ? offs[b] : 0;
      const long long p = (long long)off + i;
      if (off < 0 || off >= bs || p >= (long long)mb * bs) {
        if (lane == 0) set_error(err, kErrCapacity);
        continue;
      }
      const int blk = bt[(long long)b * mb + p / bs];
      if (blk < 0 || blk >= num_blocks) {
        if (lane == 0) set_error(err, kErrIndex);
        continue;
      }
      const long long src = row_offset(blk, layer, (int)(p % bs), L, bs, row_bytes);
      const long long dst = r * (long long)row_bytes;
      copy_row_pair(k_out + dst, kc + src, v_out + dst, vc + src, row_vecs, lane);
    }
  }
}

// ---------------------------------------------------------------------------
// validation (validate mode only): index inputs, never the pools
// ---------------------------------------------------------------------------
__global__ void validate_tables_kernel(const int32_t* __restrict__ bt, int mb,
                                       const int32_t* __restrict__ lens,
                                       const int32_t* __restrict__ offs, int batch,
                                       const int64_t* __restrict__ cu, long long total,
                                       long long num_blocks, int bs, int* err) {
  griddep_wait();
  griddep_launch_dependents();
  for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < batch; b += gridDim.x * blockDim.x) {
    const int off = offs ? offs[b] : 0;
    const int len = lens ? lens[b] : 0;
    if (off < 0 || off >= bs || len < 0 || (long long)off + len > (long long)mb * bs) {
      set_error(err, kErrCapacity);
      continue;
    }
    const long long nblk = len > 0 ? ((long long)off + len + bs - 1) / bs : 0;
    for (long long k = 0; k < nblk; ++k) {
      const int blk = bt[(long long)b * mb + k];
      if (blk < 0 || blk >= num_blocks) {
        set_error(err, kErrIndex);
        break;
      }
    }
    if (cu) {
      if (cu[b + 1] - cu[b] != len) set_error(err, kErrIndex);
      if (b == 0 && cu[0] != 0) set_error(err, kErrIndex);
      if (b == batch - 1 && cu[batch] != total) set_error(err, kErrIndex);
    }
  }
}

// Shared-prefix decode: every sequence's table agrees with row 0 on each of
// the first prefix_blocks entries it spans.
__global__ void validate_prefix_kernel(const int32_t* __restrict__ bt, int mb,
                                       const int32_t* __restrict__ lens,
                                       const int32_t* __restrict__ offs, int batch,
                                       int prefix_blocks, long long num_blocks, int bs,
                                       int* err) {
  griddep_wait();
  griddep_launch_dependents();
  // row 0 names every prefix block
  if (blockIdx.x == 0 && threadIdx.x == 0)
    for (int k = 0; k < prefix_blocks; ++k)
      if (bt[k] < 0 || bt[k] >= num_blocks) {
        set_error(err, kErrIndex);
        break;
      }
  for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < batch; b += gridDim.x * blockDim.x) {
    const int off = offs ? offs[b] : 0;
    const int len = lens[b];
    if (off < 0 || off >= bs || len < 0 || (long long)off + len > (long long)mb * bs) continue;
    const long long nblk = len > 0 ? ((long long)off + len + bs - 1) / bs : 0;
    const long long n = nblk < prefix_blocks ? nblk : prefix_blocks;
    for (long long k = 0; k < n; ++k) {
      if (bt[(long long)b * mb + k] != bt[k]) {
        set_error(err, kErrIndex);
        break;
      }
    }
  }
}

__global__ void validate_slots_kernel(const int64_t* __restrict__ slots, long long n,
                                      long long limit, int* err) {
  griddep_wait();
  griddep_launch_dependents();
  for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < n;
       t += (long long)gridDim.x * blockDim.x) {
    const int64_t s = slots[t];
    if (s < -1 || s >= limit) set_error(err, kErrIndex);
  }
}

__global__ void validate_tokens_kernel(const int32_t* __restrict__ bt, int mb,
                                       const int32_t* __restrict__ offs, int batch,
                                       const int32_t* __restrict__ tok_seq,
                                       const int32_t* __restrict__ tok_pos, long long n,
                                       long long num_blocks, int bs, int* err) {
  griddep_wait();
  griddep_launch_dependents();
  for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < n;
       t += (long long)gridDim.x * blockDim.x) {
    const int b = tok_seq[t];
    if (b < 0) continue;
    if (b >= batch) { set_error(err, kErrIndex); continue; }
    const int off = offs ? offs[b] : 0;
    if (off < 0 || off >= bs) { set_error(err, kErrCapacity); continue; }
    const long long p = (long long)off + tok_pos[t];
    if (tok_pos[t] < 0 || p >= (long long)mb * bs) { set_error(err, kErrCapacity); continue; }
    const int blk = bt[(long long)b * mb + p / bs];
    if (blk < 0 || blk >= num_blocks) set_error(err, kErrIndex);
  }
}

int grid_for(long long items, int per_block, int cap) {
  long long g = (items + per_block - 1) / per_block;
  if (g < 1) g = 1;
  if (g > cap) g = cap;
  return (int)g;
}

}  // namespace

cudaError_t launch_slot_mapping(const PoolView& p, const int32_t* bt, int mb, const int32_t* offs,
                                int batch, const int32_t* tok_seq, const int32_t* tok_pos,
                                long long n, int64_t* slots, int* err, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  SlotSrc ss{nullptr, bt, offs, tok_seq, tok_pos, slots, mb, batch};
  return launch_kernel(slot_mapping_kernel, dim3(grid_for(n, 256, 1 << 20)), dim3(256), 0, s, true,
                       ss, n, p.num_blocks, p.block_size, err);
}

namespace {

// The scatter, with slots read (FUSED false) or computed from the tokens.
template <bool FUSED>
cudaError_t launch_scatter(const PoolView& p, int layer, const void* k_new, const void* v_new,
                           const SlotSrc& ss, long long n, int* err, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  if (p.quant) {
    const dim3 grid(grid_for(n * p.num_kv_heads, kCopyWarps, 1 << 24));
    const auto* kn = static_cast<const __nv_bfloat16*>(k_new);
    const auto* vn = static_cast<const __nv_bfloat16*>(v_new);
#define PKV_QUANT_LAUNCH(VPL)                                                                  \
  launch_kernel(quant_write_slots_kernel<VPL, FUSED>, grid, dim3(kCopyThreads), 0, s, true,    \
                p.k_mut, p.v_mut, kn, vn, ss, n, p.num_blocks, p.num_layers, layer,            \
                p.block_size, p.row_bytes, p.num_kv_heads, p.scale_off, err)
    switch (p.head_dim) {
      case 32: return PKV_QUANT_LAUNCH(1);
      case 64: return PKV_QUANT_LAUNCH(2);
      case 128: return PKV_QUANT_LAUNCH(4);
      case 256: return PKV_QUANT_LAUNCH(8);
    }
#undef PKV_QUANT_LAUNCH
    return cudaErrorInvalidValue;
  }
  return launch_kernel(write_slots_kernel<FUSED>, dim3(grid_for(n, kCopyWarps, 1 << 24)),
                       dim3(kCopyThreads), 0, s, true, p.k_mut, p.v_mut,
                       static_cast<const char*>(k_new), static_cast<const char*>(v_new), ss, n,
                       p.num_blocks, p.num_layers, layer, p.block_size, p.row_bytes, err);
}

}  // namespace

cudaError_t launch_write_slots(const PoolView& p, int layer, const void* k_new, const void* v_new,
                               const int64_t* slots, long long n, int* err, int sm_count,
                               cudaStream_t s) {
  (void)sm_count;
  SlotSrc ss{slots, nullptr, nullptr, nullptr, nullptr, nullptr, 0, 0};
  return launch_scatter<false>(p, layer, k_new, v_new, ss, n, err, s);
}

cudaError_t launch_append(const PoolView& p, int layer, const int32_t* bt, int mb,
                          const int32_t* offs, int batch, const int32_t* tok_seq,
                          const int32_t* tok_pos, long long n, const void* k_new,
                          const void* v_new, int64_t* slots_out, int* err, cudaStream_t s) {
  SlotSrc ss{nullptr, bt, offs, tok_seq, tok_pos, slots_out, mb, batch};
  return launch_scatter<true>(p, layer, k_new, v_new, ss, n, err, s);
}

cudaError_t launch_gather(const PoolView& p, int layer, const int32_t* bt, int mb,
                          const int32_t* offs, int batch, const int64_t* cu, long long total,
                          void* k_out, void* v_out, int* err, cudaStream_t s) {
  if (total == 0 || batch == 0) return cudaSuccess;
  const long long groups = (total + kGatherRows - 1) / kGatherRows;
  return launch_kernel(gather_kernel, dim3(grid_for(groups, kCopyWarps, 1 << 24)),
                       dim3(kCopyThreads), 0, s, true, p.k, p.v, bt, mb, offs, batch, cu, total,
                       static_cast<char*>(k_out), static_cast<char*>(v_out), p.num_blocks,
                       p.num_layers, layer, p.block_size, p.row_bytes, err);
}

cudaError_t launch_validate_tables(const PoolView& p, const int32_t* bt, int mb,
                                   const int32_t* lens, const int32_t* offs, int batch,
                                   const int64_t* cu, long long total, int* err, cudaStream_t s) {
  if (batch == 0) return cudaSuccess;
  validate_tables_kernel<<<grid_for(batch, 128, 4096), 128, 0, s>>>(
      bt, mb, lens, offs, batch, cu, total, p.num_blocks, p.block_size, err);
  return cudaGetLastError();
}

cudaError_t launch_validate_prefix(const PoolView& p, const int32_t* bt, int mb,
                                   const int32_t* lens, const int32_t* offs, int batch,
                                   int prefix_blocks, int* err, cudaStream_t s) {
  if (batch == 0 || prefix_blocks == 0) return cudaSuccess;
  validate_prefix_kernel<<<grid_for(batch, 128, 4096), 128, 0, s>>>(
      bt, mb, lens, offs, batch, prefix_blocks, p.num_blocks, p.block_size, err);
  return cudaGetLastError();
}

cudaError_t launch_validate_slots(const PoolView& p, const int64_t* slots, long long n, int* err,
                                  cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  validate_slots_kernel<<<grid_for(n, 256, 1 << 20), 256, 0, s>>>(
      slots, n, p.num_blocks * p.block_size, err);
  return cudaGetLastError();
}

cudaError_t launch_validate_tokens(const PoolView& p, const int32_t* bt, int mb,
                                   const int32_t* offs, int batch, const int32_t* tok_seq,
                                   const int32_t* tok_pos, long long n, int* err, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  validate_tokens_kernel<<<grid_for(n, 256, 1 << 20), 256, 0, s>>>(
      bt, mb, offs, batch, tok_seq, tok_pos, n, p.num_blocks, p.block_size, err);
  return cudaGetLastError();
}

}  // namespace pkv
