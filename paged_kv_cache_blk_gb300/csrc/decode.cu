// Paged decode attention: split-K partial pass + combine pass.
//
// What is computed ("step14_2 - index_select gather", comparison with vLLM;
// "vLLM PagedAttention source notes" §2.3; mini-runtime ch.12 §3.1): for each
// sequence b and query head h (kv head g = h / (Hq/Hkv)), attention of the one
// query over the seq_len[b] K/V rows that the block table names, read in place
// from the pool; no contiguous copy of K/V is ever made.
//
// Design (GB300, one GPU):
//  * Work is the flat list of (sequence, logical block) pairs of the batch in
//    order.  A persistent grid of `grid` CTAs (one per SM by default) splits
//    that list into equal contiguous ranges, so every CTA streams the same
//    number of blocks whatever the length mix.  A CTA range cuts sequences
//    into segments; the segment of sequence b inside CTA c has index c + b
//    (unique because both the ranges and the sequences are in order).
//  * Inside a CTA one producer warp streams the K and V rows of each block
//    into a ring of shared-memory stages, completion counted on an mbarrier.
//    bf16 pools: per stage, tensor copies (cp.async.bulk.tensor) of boxes of
//    64 elements x the stage's token rows x all kv heads, K then V, with the
//    128-byte swizzle, so the 8 rows an ldmatrix reads fall in 8 different
//    bank groups.  Four copies move a 16-row stage (64 KB for Hkv 8, D 128):
//    far fewer requests than one copy per row, which is what bounded the
//    per-SM rate of row copies.  int8 pools: the same with code and scale
//    boxes.  fp32 pools: the 32 lanes issue one bulk copy (cp.async.bulk) per
//    token row, each landing in a row padded by 16 bytes.  A stage starts at
//    the sequence's first row in the block (the first-block offset) and the
//    consumers use only the rows the sequence covers; a box may carry rows
//    past them, which are never used (past the pool they arrive as zeros).
//  * Eight consumer warps compute; warp w serves kv head w % Hkv for all
//    G = Hq/Hkv query heads of that group, so each K/V byte is read from HBM
//    once and used by all G heads (GQA grouping).
//      bf16 pools: tensor cores (mma.sync m16n8k16, fp32 accumulate).
//        S^T[t][h] = K[t][:] . Q[h][:] with the 16 tokens of a stage as M and
//        the G heads as N (8 columns); online softmax in registers (exp2 of
//        pre-scaled scores); P^T goes to shared memory as bf16 and
//        O^T[d][h] += V^T[d][t] P^T[t][h] with d as M.  About 110
//        instructions per (stage, head) keep the SM far below its issue rate,
//        so the copy pipeline alone sets the speed.
//      fp32 pools: CUDA-core FMAs in fp32 (8 lanes per token for Q.K with a
//        butterfly that sums and spreads the G scores; each lane owns D/32
//        output elements for PV).
//  * At a segment end the warp either writes the normalised output (sequence
//    entirely inside this CTA) or the partial state (m, l, acc) to the
//    workspace; the combine kernel merges partial states with the log-sum-exp
//    rule  out = sum_c 2^(m_c-M) acc_c / sum_c 2^(m_c-M) l_c.
//  * Every mbarrier wait is bounded (mbar_wait), and once one CTA gives up the
//    pending waits of every other CTA leave too.  A wait that gives up sets
//    the error word and the warp leaves; the producer always waits for every
//    copy it issued to land before it returns, so no CTA exits with a copy
//    into its shared memory still in flight.
#include <cfloat>
#include <cmath>
#include <cstring>
#include <type_traits>

#include <cuda_fp16.h>

#include "common.cuh"
#include "quant.cuh"
#include "tma.cuh"

namespace pkv {
namespace {

constexpr int kNW = 8;     // consumer warps (bf16 / fp32 pools)
constexpr int kNWI8 = 8;   // consumer warps (int8 pools)

// consumer warps of the kernel instance for element type T
template <typename T>
__host__ __device__ constexpr int consumer_warps() { return sizeof(T) == 1 ? kNWI8 : kNW; }
constexpr int kMaxStageTokens = 16;       // rows per stage (one mma M tile)
constexpr int kMaxPW = kMaxStageTokens / 4;
constexpr int kMaxStages = 8;
constexpr int kRowPad = 16;               // bytes of padding after each staged row
constexpr float kLog2e = 1.4426950408889634f;
constexpr unsigned kFull = 0xffffffffu;

enum : int { kStart = 1, kEnd = 2, kLast = 4, kSingle = 8 };

// Kernel modes: plain decode attention, the fused decode step (new rows
// stored first), and the suffix pass of shared-prefix decode (the table
// entries after the shared prefix; every state goes to the workspace).
enum : int { kModePlain = 0, kModeStep = 1, kModeSuffix = 2 };

struct Params {
  const char* k_base;  // block 0, this layer, row 0
  const char* v_base;
  long long block_stride;  // bytes from one block to the next (L * bs * row_bytes)
  long long num_blocks;
  const void* q;
  void* out;
  const int32_t* bt;
  const int32_t* lens;
  const int32_t* offs;
  float* ws_acc;
  float* ws_ml;
  long long* ws_cu;
  long long* ws_meta;
  int* err;
  int mb, batch, hq, hkv, bs, row_bytes, rs, st, stages;
  int nw;       // consumer warps (the producer is warp nw)
  int mstride;  // floats between two warps' merge buffers
  int stage_bytes;  // bytes of one pipeline stage (a multiple of 1024)
  // int8 pools: stage carve (K codes, V codes, K scales, V scales), the bytes
  // the four tensor copies of a stage deliver, the scale bytes of a row, the
  // pitch of a warp's fp16 V tile, and the token-row coordinate of a block
  int off_kc, off_vc, off_ks, off_vs, tx_bytes, sbytes, vrs;
  // bf16 pools: rows per tensor-copy box, bytes of one box, 64-element halves
  // of a head row (the K boxes of a stage, then the V boxes)
  int box_rows, box_bytes, halves;
  long long rows_per_block;  // num_layers * block_size
  int layer_row;             // layer * block_size
  float qscale;
  // shared-memory carve (bytes from the start of dynamic smem)
  int off_bar, off_desc, off_cu, off_scan, off_pbuf, off_mbuf, off_vbuf;
  // fused decode step: the new row of sequence b is k_new / v_new +
  // b * new_row_bytes (Hkv * D elements of q's dtype), stored into the pool
  // through k_out / v_out (block 0, this layer, row 0); int8 pools quantise
  // it (scales at byte scale_off of the row)
  const char* k_new;
  const char* v_new;
  char* k_out;
  char* v_out;
  int new_row_bytes;
  int scale_off;
  int prefix_blocks;  // shared-prefix suffix pass: table entries of the shared prefix
  unsigned long long wait_ns;  // bound of one wait (0 = the default)
  int epoch;  // this launch's number (see WaitCtl)
  int skip_fill;  // test hook: 1 = CTA 0, 2 = every CTA stalls its consumers
};

// Tensor maps of an int8 pool (unused for bf16 / fp32 pools): K and V codes
// as (d, token row, kv head) boxes of (D, stage tokens, Hkv) bytes with the
// D-byte swizzle, and the scale bytes as (byte, token row) boxes.
struct I8Maps {
  CUtensorMap kc, vc, ks, vs;
};

// ---- small helpers ----------------------------------------------------------

template <typename T>
__device__ __forceinline__ void widen16(const uint4& r, float* f) {
  if constexpr (sizeof(T) == 2) {
    f[0] = bf16_lo(r.x); f[1] = bf16_hi(r.x); f[2] = bf16_lo(r.y); f[3] = bf16_hi(r.y);
    f[4] = bf16_lo(r.z); f[5] = bf16_hi(r.z); f[6] = bf16_lo(r.w); f[7] = bf16_hi(r.w);
  } else {
    f[0] = __uint_as_float(r.x); f[1] = __uint_as_float(r.y);
    f[2] = __uint_as_float(r.z); f[3] = __uint_as_float(r.w);
  }
}

template <typename T, int PVE>
__device__ __forceinline__ void load_pv(const char* p, float (&f)[PVE]) {
  if constexpr (sizeof(T) == 2) {
    if constexpr (PVE == 4) {
      const uint2 r = *reinterpret_cast<const uint2*>(p);
      f[0] = bf16_lo(r.x); f[1] = bf16_hi(r.x); f[2] = bf16_lo(r.y); f[3] = bf16_hi(r.y);
    } else {
      const uint32_t r = *reinterpret_cast<const uint32_t*>(p);
      f[0] = bf16_lo(r); f[1] = bf16_hi(r);
    }
  } else {
    if constexpr (PVE == 4) {
      const float4 r = *reinterpret_cast<const float4*>(p);
      f[0] = r.x; f[1] = r.y; f[2] = r.z; f[3] = r.w;
    } else {
      const float2 r = *reinterpret_cast<const float2*>(p);
      f[0] = r.x; f[1] = r.y;
    }
  }
}

// Stores of the split-K states and the block prefix sums, which the combine
// reads after the whole K/V stream has passed through L2: the evict_last
// policy keeps them there instead of letting the stream push them to DRAM.
__device__ __forceinline__ uint64_t l2_keep_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void st_keep(float* a, float v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(a), "f"(v), "l"(pol)
               : "memory");
}

__device__ __forceinline__ void st_keep(long long* a, long long v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.s64 [%0], %1, %2;" ::"l"(a), "l"(v), "l"(pol)
               : "memory");
}

template <typename T>
__device__ __forceinline__ void store_elem(void* base, long long idx, float x) {
  if constexpr (sizeof(T) == 2) {
    static_cast<__nv_bfloat16*>(base)[idx] = __float2bfloat16_rn(x);
  } else {
    static_cast<float*>(base)[idx] = x;
  }
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void ldsm_x2_t(uint32_t (&r)[2], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(addr)
               : "memory");
}

// Transposing load of a 16 x 16 byte matrix (rows addressed by lanes 0-15):
// lane l receives column l/4 (r0) and column l/4 + 8 (r1) of rows
// 4 (l % 4) .. 4 (l % 4) + 3, one byte per row, lowest row in the low byte.
__device__ __forceinline__ void ldsm_b8_t(uint32_t& r0, uint32_t& r1, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m16n16.x1.trans.shared.b8 {%0,%1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(addr)
               : "memory");
}

// D[16x8] += A[16x16] * B[16x8], bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Sum partial dot products over the 8 lanes of a token group while spreading
// the G heads over them: each step either halves the heads a lane holds
// (keeping one half, sending the other) or, once a lane holds one head, adds
// its partner's copy.  At the end lane i (within the group) holds the full
// score of head i >> (3 - log2 G).
template <int G>
__device__ __forceinline__ float butterfly(float (&v)[G], int lane) {
#pragma unroll
  for (int step = 0; step < 3; ++step) {
    const int m = 4 >> step;
    const int nh = (G >> step) > 1 ? (G >> step) : 1;  // heads held before this step
    if (nh > 1) {
      const int half = nh / 2;
      const bool upper = (lane & m) != 0;
#pragma unroll
      for (int x = 0; x < half; ++x) {
        const float send = upper ? v[x] : v[x + half];
        const float keep = upper ? v[x + half] : v[x];
        v[x] = keep + __shfl_xor_sync(kFull, send, m);
      }
    } else {
      v[0] += __shfl_xor_sync(kFull, v[0], m);
    }
  }
  return v[0];
}

// Blocks spanned by sequence b; 0 for an empty or invalid sequence (reported
// by CTA 0 only, so the error word is touched once per launch).
template <int MODE>
__device__ __forceinline__ long long seq_blocks(const Params& p, int b, bool report) {
  const int len = p.lens[b];
  const int off = p.offs ? p.offs[b] : 0;
  if (len < 0 || off < 0 || off >= p.bs || (long long)off + len > (long long)p.mb * p.bs) {
    if (report) set_error(p.err, kErrCapacity);
    return 0;
  }
  if (len == 0) return 0;
  const long long nb = ((long long)off + len + p.bs - 1) / p.bs;
  if constexpr (MODE == kModeSuffix) return nb > p.prefix_blocks ? nb - p.prefix_blocks : 0;
  return nb;
}

// Shared-memory pipeline handles.
struct Pipe {
  unsigned char* smem;
  int4* desc;
  uint32_t bar0;
  int stages;
  int stage_bytes;
  __device__ uint32_t full(int s) const { return bar0 + 8u * s; }
  __device__ uint32_t empty(int s) const { return bar0 + 8u * (stages + s); }
  __device__ uint32_t group() const { return bar0 + 8u * (2 * stages); }
  // never arrived at: the test hook's stalled wait
  __device__ uint32_t stall() const { return bar0 + 8u * (2 * stages + 1); }
};

// Reusable barrier over the consumer warps (mbarrier with nw arrivals),
// bounded like every other wait.
__device__ __forceinline__ bool group_sync(const Pipe& pp, uint32_t& gph, int lane,
                                           const WaitCtl& w) {
  __syncwarp();
  if (lane == 0) mbar_arrive(pp.group());
  const bool ok = mbar_wait(pp.group(), gph, w);
  gph ^= 1;
  return ok;
}

// ---- producer warp -----------------------------------------------------------

// Table entries, first-block offsets and lengths of 32 consecutive blocks of
// the flat list, one block per lane: loaded one batch ahead of their use, so
// their global-load latency overlaps the stages of the batch before.
struct Lookup {
  int bl;           // sequence of this lane's block
  long long j, nb;  // its index in the sequence, the sequence's block count
  int blk, off, len;
};

template <int MODE>
__device__ __forceinline__ Lookup lookup_batch(const Params& p, const long long* s_cu, int lane,
                                               long long base, long long x1, int bseq) {
  Lookup L;
  const long long xl = base + lane;
  const bool valid = xl < x1;
  int bl = bseq;
  if (valid) while (s_cu[bl + 1] <= xl) ++bl;
  L.bl = bl;
  L.j = valid ? xl - s_cu[bl] : 0;
  L.nb = s_cu[bl + 1] - s_cu[bl];
  L.blk = valid ? __ldg(p.bt + (long long)bl * p.mb + L.j) : 0;
  L.off = valid && p.offs ? __ldg(p.offs + bl) : 0;
  L.len = valid ? __ldg(p.lens + bl) : 0;
  if constexpr (MODE == kModeSuffix) {
    // the blocks after the shared prefix, read from row 0 of the block: the
    // suffix starts on a fresh block
    L.blk = valid ? __ldg(p.bt + (long long)bl * p.mb + p.prefix_blocks + L.j) : 0;
    L.len = L.off + L.len - p.prefix_blocks * p.bs;
    L.off = 0;
  }
  return L;
}

// Staging of a stage: one bulk copy per token row (fp32 pools), or tensor
// copies of whole boxes (int8 pools: codes and scales; bf16 pools: swizzled
// halves of the head rows).
enum : int { kStageRows = 0, kStageI8 = 1, kStageBf16 = 2 };

template <int STG, int MODE>
__device__ void run_producer(const Params& p, const Pipe& pp, const I8Maps& maps,
                             const long long* s_cu, int lane, long long x0, long long x1) {
  const WaitCtl w = make_wait_ctl(p.err, p.wait_ns, p.epoch);
  const int B = p.batch;
  const int ST = p.st;
  int lo = 0, hi = B;  // sequence holding block x0: largest b with s_cu[b] <= x0
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_cu[mid] <= x0) lo = mid; else hi = mid;
  }
  int bseq = lo;
  while (s_cu[bseq + 1] <= x0) ++bseq;  // skip empty sequences
  int s = 0;
  uint32_t ph = 1;  // "empty" waits start on the already completed phase
  uint32_t filled = 0, fill_par = 0;
  bool ok = true;
  const int r_lane = lane & 15;
  const bool v_lane = lane >= 16;
  const uint32_t dst_lane = smem_addr(pp.smem) + (v_lane ? ST * p.rs : 0) + r_lane * p.rs;
  const char* src_lane = (v_lane ? p.v_base : p.k_base) + (long long)r_lane * p.row_bytes;
  Lookup nxt = lookup_batch<MODE>(p, s_cu, lane, x0, x1, bseq);
  for (long long base = x0; base < x1 && ok; base += 32) {
    // this batch of 32 blocks (looked up one batch ago); then start the
    // next batch's loads
    const Lookup cur = nxt;
    const int cnt = (int)min((long long)32, x1 - base);
    if (base + 32 < x1)
      nxt = lookup_batch<MODE>(p, s_cu, lane, base + 32, x1,
                               __shfl_sync(kFull, cur.bl, cnt - 1));
    int r0 = 0, r1 = p.bs;
    if (cur.j == 0) r0 = cur.off;
    if (cur.j == cur.nb - 1) r1 = (int)(((long long)cur.off + cur.len - 1) % p.bs) + 1;
    for (int k = 0; k < cnt && ok; ++k) {
      const int kb = __shfl_sync(kFull, cur.bl, k);
      const int kblk = __shfl_sync(kFull, cur.blk, k);
      const int kr0 = __shfl_sync(kFull, r0, k);
      const int kr1 = __shfl_sync(kFull, r1, k);
      const long long kj = __shfl_sync(kFull, cur.j, k);
      const long long knb = __shfl_sync(kFull, cur.nb, k);
      const long long kx = base + k;
      const bool blk_ok = kblk >= 0 && (long long)kblk < p.num_blocks;
      if (!blk_ok && lane == 0) set_error(p.err, kErrIndex);
      const bool seg_start = (kj == 0) || (kx == x0);
      const bool seg_end = (kj == knb - 1) || (kx == x1 - 1);
      // a sequence wholly inside this CTA is finished here, unless its
      // shared-prefix state still has to be merged in
      const bool single = MODE != kModeSuffix && s_cu[kb] >= x0 && s_cu[kb + 1] <= x1;
      const char* blk_src = src_lane + (long long)kblk * p.block_stride;
      for (int rs0 = kr0; rs0 < kr1;) {
        const int re = min(kr1, (rs0 / ST + 1) * ST);
        const int n = re - rs0;
        int flags = 0;
        if (seg_start && rs0 == kr0) flags |= kStart;
        if (seg_end && re == kr1) flags |= kEnd;
        if (kx == x1 - 1 && re == kr1) flags |= kLast;
        if (single) flags |= kSingle;
        const int4 desc = make_int4(kb, blk_ok ? n : 0, flags, (int)blockIdx.x + kb);
        const uint32_t full = pp.full(s);
        const uint32_t stage = (uint32_t)s * pp.stage_bytes;
        if constexpr (STG == kStageI8) {
          // int8 pools: the consumers are the slower side, so the producer
          // mostly waits here; it sleeps rather than polls, leaving the issue
          // slots of its SMSP to the two consumer warps beside it
          if (!mbar_wait_sleep(pp.empty(s), ph, w)) { ok = false; break; }
        } else {
          if (!mbar_wait(pp.empty(s), ph, w)) { ok = false; break; }
        }
        if constexpr (STG == kStageBf16) {
          // bf16 pools: for each 64-element half of the head rows, one box of
          // (64, box_rows, Hkv) from K and one from V, starting at row rs0;
          // rows past n are masked (past the pool they arrive as zeros)
          if (lane == 0) {
            pp.desc[s] = desc;
            if (blk_ok) {
              mbar_arrive_expect_tx(full, (uint32_t)p.tx_bytes);
              const int row = (int)(kblk * p.rows_per_block + p.layer_row + rs0);
              const uint32_t base_s = smem_addr(pp.smem) + stage;
              for (int h = 0; h < p.halves; ++h) {
                tma_3d(base_s + h * p.box_bytes, &maps.kc, 64 * h, row, 0, full);
                tma_3d(base_s + (p.halves + h) * p.box_bytes, &maps.vc, 64 * h, row, 0, full);
              }
            } else {
              mbar_arrive(full);
            }
          }
        } else if constexpr (STG == kStageI8) {
          // int8 pools: four tensor copies per stage (K and V codes, K and V
          // scales), always whole boxes of st rows starting at row rs0; rows
          // past n are never read (past the pool they arrive as zeros)
          if (lane == 0) {
            pp.desc[s] = desc;
            if (blk_ok) {
              mbar_arrive_expect_tx(full, (uint32_t)p.tx_bytes);
              const int row = (int)(kblk * p.rows_per_block + p.layer_row + rs0);
              const uint32_t base_s = smem_addr(pp.smem) + stage;
              tma_3d(base_s + p.off_kc, &maps.kc, 0, row, 0, full);
              tma_3d(base_s + p.off_vc, &maps.vc, 0, row, 0, full);
              tma_2d(base_s + p.off_ks, &maps.ks, 0, row, full);
              tma_2d(base_s + p.off_vs, &maps.vs, 0, row, full);
            } else {
              mbar_arrive(full);
            }
          }
        } else {
          // lane 0 posts the stage's byte count while lanes 0-15 (K) and
          // 16-31 (V) issue one row copy each: a copy that completes before
          // the count is posted drives the count below zero for a moment,
          // and the phase cannot complete before lane 0's arrival
          if (lane == 0) {
            pp.desc[s] = desc;
            if (blk_ok) mbar_arrive_expect_tx(full, 2u * n * p.row_bytes);
            else mbar_arrive(full);
          }
          if (blk_ok && r_lane < n)
            bulk_g2s(dst_lane + stage, blk_src + (long long)rs0 * p.row_bytes, p.row_bytes, full);
        }
        __syncwarp();
        filled |= 1u << s;
        fill_par = (fill_par & ~(1u << s)) | (((ph ^ 1u) & 1u) << s);
        if (++s == pp.stages) { s = 0; ph ^= 1; }
        rs0 = re;
      }
    }
  }
  // Let every copy already issued land before the CTA (and its shared memory)
  // may go away: the consumers normally waited for them all, but consumers
  // that gave up did not.  Each stage holds at most one fill in flight (a
  // stage is refilled only after its consumers released it).
  for (int t = 0; t < pp.stages; ++t)
    if (filled & (1u << t)) mbar_wait_drain(pp.full(t), (fill_par >> t) & 1u, p.err);
  (void)ok;
}

// End of a segment for the tensor-core consumers: sum the row shares of l,
// merge the warps that served the same kv head (when Hkv < 8), then write the
// normalised output (sequence inside one CTA) or the partial state (m, l, acc)
// to the workspace.  False when a bounded wait gave up.
template <int D, int G>
__device__ __forceinline__ bool mma_segment_end(const Params& p, const Pipe& pp, uint32_t& gph,
                                                float (&o)[D / 16][4], float m0, float m1,
                                                float l0, float l1, bool mv, int b, int seg,
                                                int flags, int warp, int lane,
                                                const WaitCtl& w) {
  constexpr int KS = D / 16;
  const int hkv = p.hkv;
  const int g = warp % hkv;
  const int wsub = warp / hkv;
  const int wph = p.nw / hkv;
  const int gl = lane >> 2;
  const int qi = lane & 3;
  float* mbuf = reinterpret_cast<float*>(pp.smem + p.off_mbuf);
  // row sums: each thread held the share of its token rows
  float L0 = l0, L1 = l1;
#pragma unroll
  for (int o2 = 4; o2 < 32; o2 <<= 1) {
    L0 += __shfl_xor_sync(kFull, L0, o2);
    L1 += __shfl_xor_sync(kFull, L1, o2);
  }
  float M0 = mv ? m0 : -INFINITY, M1 = mv ? m1 : -INFINITY;
  const int h0 = 2 * qi, h1 = h0 + 1;
  if (wph > 1) {
    // merge the token shares of the warps serving the same kv head
    float* mw = mbuf + warp * p.mstride;
#pragma unroll
    for (int kt = 0; kt < KS; ++kt) {
      const int d0 = kt * 16 + gl, d1 = d0 + 8;
      if (h0 < G) { mw[h0 * (D + 2) + d0] = o[kt][0]; mw[h0 * (D + 2) + d1] = o[kt][2]; }
      if (h1 < G) { mw[h1 * (D + 2) + d0] = o[kt][1]; mw[h1 * (D + 2) + d1] = o[kt][3]; }
    }
    if (gl == 0) {
      if (h0 < G) { mw[h0 * (D + 2) + D] = M0; mw[h0 * (D + 2) + D + 1] = L0; }
      if (h1 < G) { mw[h1 * (D + 2) + D] = M1; mw[h1 * (D + 2) + D + 1] = L1; }
    }
    if (!group_sync(pp, gph, lane, w)) return false;
    if (wsub == 0) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int h = h0 + hh;
        if (h >= G) continue;
        float Mx = -INFINITY;
        for (int w2 = g; w2 < p.nw; w2 += hkv)
          Mx = fmaxf(Mx, mbuf[w2 * p.mstride + h * (D + 2) + D]);
        float Ls = 0.f;
        float acc[KS][2];
#pragma unroll
        for (int kt = 0; kt < KS; ++kt) acc[kt][0] = acc[kt][1] = 0.f;
        if (Mx != -INFINITY) {
          for (int w2 = g; w2 < p.nw; w2 += hkv) {
            const float* src = mbuf + w2 * p.mstride + h * (D + 2);
            if (src[D] == -INFINITY) continue;
            const float wgt = exp2f(src[D] - Mx);
            Ls += wgt * src[D + 1];
#pragma unroll
            for (int kt = 0; kt < KS; ++kt) {
              acc[kt][0] += wgt * src[kt * 16 + gl];
              acc[kt][1] += wgt * src[kt * 16 + gl + 8];
            }
          }
        }
#pragma unroll
        for (int kt = 0; kt < KS; ++kt) {
          o[kt][hh] = acc[kt][0];
          o[kt][2 + hh] = acc[kt][1];
        }
        if (hh == 0) { M0 = Mx; L0 = Ls; } else { M1 = Mx; L1 = Ls; }
      }
    }
    if (!group_sync(pp, gph, lane, w)) return false;
  }
  if (wsub == 0) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int h = h0 + hh;
      if (h >= G) continue;
      const float Lh = hh == 0 ? L0 : L1;
      const float Mh = hh == 0 ? M0 : M1;
      const long long row_out = (long long)b * p.hq + g * G + h;
      const long long row_ws = (long long)seg * p.hq + g * G + h;
      if (flags & kSingle) {
        const float inv = Lh > 0.f ? 1.f / Lh : 0.f;
#pragma unroll
        for (int kt = 0; kt < KS; ++kt) {
          store_elem<__nv_bfloat16>(p.out, row_out * D + kt * 16 + gl,
                                    o[kt][hh] * inv);
          store_elem<__nv_bfloat16>(p.out, row_out * D + kt * 16 + gl + 8,
                                    o[kt][2 + hh] * inv);
        }
      } else {
        const uint64_t pol = l2_keep_policy();
#pragma unroll
        for (int kt = 0; kt < KS; ++kt) {
          st_keep(p.ws_acc + row_ws * D + kt * 16 + gl, o[kt][hh], pol);
          st_keep(p.ws_acc + row_ws * D + kt * 16 + gl + 8, o[kt][2 + hh], pol);
        }
        if (gl == 0) {
          st_keep(p.ws_ml + row_ws * 2, Mh, pol);
          st_keep(p.ws_ml + row_ws * 2 + 1, Lh, pol);
        }
      }
    }
  }
  return true;
}

// ---- bf16 consumer: tensor cores ---------------------------------------------

template <int D, int G>
__device__ void run_consumer_mma(const Params& p, const Pipe& pp, int warp, int lane) {
  const WaitCtl w = make_wait_ctl(p.err, p.wait_ns, p.epoch);
  constexpr int KS = D / 16;  // k-steps of Q.K = m-tiles of P.V
  const int hkv = p.hkv;
  const int g = warp % hkv;
  const int wsub = warp / hkv;
  const int wph = p.nw / hkv;
  const int gl = lane >> 2;  // mma group row
  const int qi = lane & 3;   // mma thread in group
  // The stage holds, per 64-element half of the head rows, a K box and then
  // a V box of Hkv x box_rows lines of 128 bytes (line g * box_rows + row),
  // written with the 128-byte swizzle: 16-byte chunk c of line L sits at
  // chunk c ^ (L & 7).  The 8 rows one ldmatrix reads are 8 consecutive
  // lines, so they fall in 8 different chunk positions: no bank conflicts.
  const int R = p.box_rows;
  const uint32_t box = p.box_bytes;
  const uint32_t v_boxes = p.halves * box;
  const int ld_t = (lane & 7) + ((lane >> 3) & 1) * 8;  // K rows (A of Q.K, non-trans)
  const int ld_c = lane >> 4;
  const int pv_t = (lane & 7) + (lane >> 4) * 8;        // V rows (A of P.V, trans)
  const int pv_c = (lane >> 3) & 1;
  unsigned char* ptile = pp.smem + p.off_pbuf + warp * 256;  // P^T [16 t][8 h] bf16
  const uint32_t pt_addr = smem_addr(ptile);
  const float qs = p.qscale;

  uint32_t qb[KS][2];
  float o[KS][4];
  float m0 = 0.f, m1 = 0.f, l0 = 0.f, l1 = 0.f;
  bool mv = false;

  int s = 0;
  uint32_t ph = 0, gph = 0;
  while (true) {
    if (!mbar_wait(pp.full(s), ph, w)) return;
    const int4 dsc = pp.desc[s];
    const int b = dsc.x, n = dsc.y, flags = dsc.z, seg = dsc.w;
    const uint32_t sbase = smem_addr(pp.smem) + (uint32_t)s * pp.stage_bytes;

    if (flags & kStart) {
      mv = false;
      m0 = m1 = l0 = l1 = 0.f;
#pragma unroll
      for (int kt = 0; kt < KS; ++kt)
#pragma unroll
        for (int c = 0; c < 4; ++c) o[kt][c] = 0.f;
      // B fragments of Q^T: column gl is query head g*G + gl
      const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
          static_cast<const char*>(p.q) + (((long long)b * p.hq + g * G + gl) * D + 2 * qi) * 2);
#pragma unroll
      for (int j = 0; j < KS; ++j) {
        qb[j][0] = gl < G ? __ldg(qrow + 8 * j) : 0u;
        qb[j][1] = gl < G ? __ldg(qrow + 8 * j + 4) : 0u;
      }
    }

    for (int mt = wsub; mt * 16 < n; mt += wph) {
      const int t_lo = mt * 16;
      // rows past n hold stale data: read a valid row instead (it is masked)
      const int rk = min(t_lo + ld_t, n - 1);
      const int rv = min(t_lo + pv_t, n - 1);
      const int lk = g * R + rk, lv = g * R + rv;  // their lines in the boxes
      const uint32_t k_line = sbase + lk * 128, v_line = sbase + v_boxes + lv * 128;
      const int kx = lk & 7, vx = lv & 7;
      float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < KS; ++j) {
        // chunk 2j + ld_c of the head row: box j / 4, chunk (2j % 8) + ld_c
        uint32_t a[4];
        ldsm_x4(a, k_line + (j >> 2) * box + ((((2 * j) & 7) + ld_c) ^ kx) * 16);
        mma_bf16(sc, a, qb[j][0], qb[j][1]);
      }
      const int t0 = t_lo + gl, t1 = t0 + 8;
      sc[0] = t0 < n ? sc[0] * qs : -INFINITY;
      sc[1] = t0 < n ? sc[1] * qs : -INFINITY;
      sc[2] = t1 < n ? sc[2] * qs : -INFINITY;
      sc[3] = t1 < n ? sc[3] * qs : -INFINITY;
      float mx0 = fmaxf(sc[0], sc[2]), mx1 = fmaxf(sc[1], sc[3]);
#pragma unroll
      for (int o2 = 4; o2 < 32; o2 <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, o2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, o2));
      }
      const float n0 = mv ? fmaxf(m0, mx0) : mx0;
      const float n1 = mv ? fmaxf(m1, mx1) : mx1;
      const float a0 = mv ? exp2f(m0 - n0) : 0.f;
      const float a1 = mv ? exp2f(m1 - n1) : 0.f;
      const float p0 = exp2f(sc[0] - n0), p1 = exp2f(sc[1] - n1);
      const float p2 = exp2f(sc[2] - n0), p3 = exp2f(sc[3] - n1);
      l0 = l0 * a0 + p0 + p2;  // this thread's share; summed over rows at the end
      l1 = l1 * a1 + p1 + p3;
      m0 = n0;
      m1 = n1;
      mv = true;
#pragma unroll
      for (int kt = 0; kt < KS; ++kt) {
        o[kt][0] *= a0; o[kt][1] *= a1; o[kt][2] *= a0; o[kt][3] *= a1;
      }
      *reinterpret_cast<uint32_t*>(ptile + gl * 16 + qi * 4) = pack_bf16x2(p0, p1);
      *reinterpret_cast<uint32_t*>(ptile + (gl + 8) * 16 + qi * 4) = pack_bf16x2(p2, p3);
      __syncwarp();
      uint32_t pb[2];
      ldsm_x2_t(pb, pt_addr + (lane & 15) * 16);
#pragma unroll
      for (int kt = 0; kt < KS; ++kt) {
        uint32_t a[4];
        ldsm_x4_t(a, v_line + (kt >> 2) * box + ((((2 * kt) & 7) + pv_c) ^ vx) * 16);
        mma_bf16(o[kt], a, pb[0], pb[1]);
      }
      __syncwarp();
    }

    if (flags & kEnd) {
      if (!mma_segment_end<D, G>(p, pp, gph, o, m0, m1, l0, l1, mv, b, seg, flags, warp,
                                        lane, w))
        return;
    }

    __syncwarp();
    if (lane == 0) mbar_arrive(pp.empty(s));
    if (++s == pp.stages) { s = 0; ph ^= 1; }
    if (flags & kLast) break;
  }
}

// ---- int8 consumer: tensor cores on converted codes ----------------------------
//
// Both products run on fp16 tensor cores with fp32 accumulators; every int8
// code is exact in fp16 (|code| <= 127).
// K side.  q . (code * scale) = scale * (q . code): the A fragments of S^T
// are K's codes, the B fragments are q scaled by a power of two 2^e into
// fp16 (exact except for values below 2^-28 of the head's absmax), and the
// fp32 accumulator is multiplied by scale_k * 2^-e per (token, head).  A lane
// takes its A values from one contiguous run of D/4 codes per row: the k
// index of the mma is a fixed permutation of d applied to both operands
// (lane qi, k-step j, slots 2qi, 2qi+1, 2qi+8, 2qi+9 <-> d = (D/4) qi + 4j +
// 0..3), which leaves every dot product unchanged.
// V side.  sum_t p_t (code_t * scale_t) = sum_t (p_t scale_t) code_t: the V
// scales are folded into the softmax weights, normalised by a running power
// of two 2^E (E = the largest scale exponent seen in the segment, raised like
// the softmax maximum, with an exact power-of-two rescale of O) so that the
// fp16 weights p * scale * 2^-E stay in [0, 2); O is multiplied back by 2^E
// at the segment end.  The codes of the 16 tokens of a tile are converted to
// an fp16 tile in the warp's shared memory so the ldmatrix.trans path of the
// bf16 consumer serves unchanged.

// Four stored code bytes (offset binary: u = code + 128) -> two fp16x2
// holding code + 1152 (codes 0,1 and 2,3): each byte becomes the low mantissa
// byte of 1024 + u.  The bias is removed after the products (kBias times the
// sum of the other operand), so the conversion is two byte permutes.
constexpr float kBias = 1152.f;
constexpr uint32_t kBiasF16x2 = 0x64806480u;  // (1152, 1152) in fp16
__device__ __forceinline__ void i8x4_to_f16b(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(lo) : "r"(w), "r"(0x64646464u));
  asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(hi) : "r"(w), "r"(0x64646464u));
}

// Address of 16-byte unit u of line `line` of a code tile written by a tensor
// copy with the D-byte swizzle (tile 1024-byte aligned, D-byte lines): the
// unit index is XORed with address bits 7.. of the line (three bits for the
// 128-byte swizzle, two for the 64-byte one).
template <int D>
__device__ __forceinline__ uint32_t code_unit(uint32_t tile, int line, int u) {
  constexpr int kMask = D == 128 ? 7 : 3;
  const int x = ((line * D) >> 7) & kMask;
  return tile + line * D + ((u ^ x) << 4);
}

// Shared-memory accesses by 32-bit shared-window address (the compiler
// cannot always prove a generic pointer is shared and would then issue
// generic loads, which wait on the long scoreboard).
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "r"(a));
  return r;
}

__device__ __forceinline__ float lds_f32(uint32_t a) {
  float r;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(r) : "r"(a));
  return r;
}

__device__ __forceinline__ void sts32(uint32_t a, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// D[16x8] += A[16x16] * B[16x8], fp16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <int D, int G>
__device__ void run_consumer_i8(const Params& p, const Pipe& pp, int warp, int lane) {
  const WaitCtl w = make_wait_ctl(p.err, p.wait_ns, p.epoch);
  constexpr int KS = D / 16;  // k-steps of Q.K = m-tiles of P.V
  constexpr int QW = D / 4;   // codes (bytes) of one K row a lane reads
  const int hkv = p.hkv;
  const int g = warp % hkv;
  const int wsub = warp / hkv;
  const int wph = p.nw / hkv;
  const int gl = lane >> 2;  // mma group row
  const int qi = lane & 3;   // mma thread in group
  const int ST = p.st;
  const int sb = p.sbytes;
  // P^T tile [16 rows][8 heads] fp16; token t goes to row prow(t) (see below)
  const uint32_t pt_addr = smem_addr(pp.smem + p.off_pbuf + warp * 256);
  const uint32_t smem0 = smem_addr(pp.smem);

  uint32_t qb[KS][2];
  float qs0 = 0.f, qs1 = 0.f;  // score factors of this lane's head columns 2qi, 2qi+1
  float kb0 = 0.f, kb1 = 0.f;  // K-code bias terms of those columns: 1152 * sum(q)
  float o[KS][4];
  float vb0 = 0.f, vb1 = 0.f;  // V-code bias terms of O: 1152 * sum(weights)
  float m0 = 0.f, m1 = 0.f, l0 = 0.f, l1 = 0.f;
  bool mv = false;
  int ev = 0;  // biased exponent E of the V-weight normaliser 2^(E-127)
  float f = __uint_as_float(254u << 23);  // 2^(127-E): the weight factor
  // Offsets of this lane's code units within a stage's code tile.  Every row
  // of a tile holds real data (a tensor copy always fills all ST rows, past
  // the pool with zeros), so rows past n are read as they are: their scores
  // are masked and their weights are zero.
  //  K: rows gl and gl + 8, the lane's QW-byte run of d.
  //  V: the 16-byte unit kt of token row (lane & 15), the row address of
  //     a transposing 16 x 16 byte ldmatrix.  That load hands lane (gl, qi)
  //     bytes d = 16 kt + gl (and + 8) of tokens 4 qi .. 4 qi + 3, which
  //     after conversion are the A fragment of V^T when the k index of the
  //     P.V mma maps k = 2qi + {0, 1} to token 4qi + {0, 1} and k = 2qi + 8 +
  //     {0, 1} to token 4qi + 2 + {0, 1}; P^T is stored with the same map.
  uint32_t koff[2][QW / 16], voff[KS];
#pragma unroll
  for (int i = 0; i < QW / 16; ++i) {
    koff[0][i] = code_unit<D>(0, g * ST + gl, (QW / 16) * qi + i);
    koff[1][i] = code_unit<D>(0, g * ST + gl + 8, (QW / 16) * qi + i);
  }
#pragma unroll
  for (int kt = 0; kt < KS; ++kt) voff[kt] = code_unit<D>(0, g * ST + (lane & 15), kt);
  // P^T rows of this lane's tokens gl and gl + 8 under that map
  auto prow = [](int t) { return (t & 2) ? 2 * (t >> 2) + 8 + (t & 1) : 2 * (t >> 2) + (t & 1); };
  const uint32_t p_st0 = pt_addr + prow(gl) * 16 + qi * 4;
  const uint32_t p_st1 = pt_addr + prow(gl + 8) * 16 + qi * 4;

  int s = 0;
  uint32_t ph = 0, gph = 0;
  int turn = 0;  // the wph warps of a kv head take the stages in turn
  while (true) {
    if (!mbar_wait(pp.full(s), ph, w)) return;
    const int4 dsc = pp.desc[s];
    const int b = dsc.x, flags = dsc.z, seg = dsc.w;
    const int n = turn == wsub ? dsc.y : 0;  // rows this warp processes
    if (++turn == wph) turn = 0;
    // stage: code tiles [Hkv][ST rows][D bytes] with the D-byte swizzle,
    // scales [ST rows][sb bytes]
    const uint32_t base = smem0 + s * pp.stage_bytes;
    const uint32_t sKc = base + p.off_kc, sVc = base + p.off_vc;
    const uint32_t sKs = base + p.off_ks + 4 * g, sVs = base + p.off_vs + 4 * g;

    if (flags & kStart) {
      mv = false;
      m0 = m1 = l0 = l1 = 0.f;
      vb0 = vb1 = 0.f;
      ev = 0;
      f = __uint_as_float(254u << 23);
#pragma unroll
      for (int kt = 0; kt < KS; ++kt)
#pragma unroll
        for (int c = 0; c < 4; ++c) o[kt][c] = 0.f;
      // this lane's QW query values of head g*G + gl (zero for padding columns)
      uint4 raw[QW / 8];
      const uint4* qrow = reinterpret_cast<const uint4*>(
          static_cast<const char*>(p.q) + (((long long)b * p.hq + g * G + gl) * D + QW * qi) * 2);
#pragma unroll
      for (int i = 0; i < QW / 8; ++i) raw[i] = gl < G ? __ldg(qrow + i) : make_uint4(0, 0, 0, 0);
      // |q| maximum of the head, compared as bf16 bit patterns
      uint32_t mx = 0;
#pragma unroll
      for (int i = 0; i < QW / 8; ++i) {
        const uint32_t w[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) mx = max(mx, max(w[k] & 0x7FFFu, (w[k] >> 16) & 0x7FFFu));
      }
      mx = max(mx, __shfl_xor_sync(kFull, mx, 1));
      mx = max(mx, __shfl_xor_sync(kFull, mx, 2));
      // 2^e brings the absmax into [2^14, 2^15): fp16 holds every bf16 value
      // down to 2^-28 of it exactly
      int e = 0;
      if (mx != 0) e = min(126, max(-126, 141 - (int)((mx >> 7) & 0xFF)));
      const float up = __uint_as_float((uint32_t)(127 + e) << 23);
      const float down = __uint_as_float((uint32_t)(127 - e) << 23);
#pragma unroll
      for (int j = 0; j < KS; ++j) {
        const uint4& r = raw[j >> 1];
        const uint32_t w0 = (j & 1) ? r.z : r.x, w1 = (j & 1) ? r.w : r.y;
        qb[j][0] = pack_f16x2(bf16_lo(w0) * up, bf16_hi(w0) * up);
        qb[j][1] = pack_f16x2(bf16_lo(w1) * up, bf16_hi(w1) * up);
      }
      // sum of the fp16 query values of the head (for the K-code bias)
      float qsum = 0.f;
#pragma unroll
      for (int j = 0; j < KS; ++j) {
        const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&qb[j][0]));
        const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&qb[j][1]));
        qsum += (f0.x + f0.y) + (f1.x + f1.y);
      }
      qsum += __shfl_xor_sync(kFull, qsum, 1);
      qsum += __shfl_xor_sync(kFull, qsum, 2);
      kb0 = kBias * __shfl_sync(kFull, qsum, (2 * qi) * 4);
      kb1 = kBias * __shfl_sync(kFull, qsum, (2 * qi + 1) * 4);
      qs0 = p.qscale * __shfl_sync(kFull, down, (2 * qi) * 4);
      qs1 = p.qscale * __shfl_sync(kFull, down, (2 * qi + 1) * 4);
    }

    if (n > 0) {  // one 16-row tile (stages never hold more rows)
      const int t0 = gl, t1 = gl + 8;
      uint32_t w0[KS], w1[KS];
#pragma unroll
      for (int i = 0; i < QW / 16; ++i) {
        const uint4 a = lds128(sKc + koff[0][i]);
        const uint4 c = lds128(sKc + koff[1][i]);
        w0[4 * i] = a.x; w0[4 * i + 1] = a.y; w0[4 * i + 2] = a.z; w0[4 * i + 3] = a.w;
        w1[4 * i] = c.x; w1[4 * i + 1] = c.y; w1[4 * i + 2] = c.z; w1[4 * i + 3] = c.w;
      }
      // scales of rows past n may be anything (rows of other blocks): their
      // scores are masked below and their V scales replaced by 0
      const float sk0 = lds_f32(sKs + t0 * sb), sk1 = lds_f32(sKs + t1 * sb);
      const float sv0 = t0 < n ? lds_f32(sVs + t0 * sb) : 0.f;
      const float sv1 = t1 < n ? lds_f32(sVs + t1 * sb) : 0.f;
      // two independent accumulation chains over the k-steps
      float sa[4] = {0.f, 0.f, 0.f, 0.f}, sq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < KS; ++j) {
        uint32_t a[4];
        i8x4_to_f16b(w0[j], a[0], a[2]);
        i8x4_to_f16b(w1[j], a[1], a[3]);
        mma_f16((j & 1) ? sq : sa, a, qb[j][0], qb[j][1]);
      }
      float sc[4];
      sc[0] = t0 < n ? ((sa[0] + sq[0]) - kb0) * qs0 * sk0 : -INFINITY;
      sc[1] = t0 < n ? ((sa[1] + sq[1]) - kb1) * qs1 * sk0 : -INFINITY;
      sc[2] = t1 < n ? ((sa[2] + sq[2]) - kb0) * qs0 * sk1 : -INFINITY;
      sc[3] = t1 < n ? ((sa[3] + sq[3]) - kb1) * qs1 * sk1 : -INFINITY;
      float mx0 = fmaxf(sc[0], sc[2]), mx1 = fmaxf(sc[1], sc[3]);
      // The running maxima move only when some lane's stage maximum passes
      // them (rare after the first tiles); otherwise the reduction would
      // return them unchanged and the correction factors would be exactly 1.
      float n0 = m0, n1 = m1, a0 = 1.f, a1 = 1.f;
      if (!mv || __any_sync(kFull, mx0 > m0 || mx1 > m1)) {
#pragma unroll
        for (int o2 = 4; o2 < 32; o2 <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, o2));
          mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, o2));
        }
        n0 = mv ? fmaxf(m0, mx0) : mx0;
        n1 = mv ? fmaxf(m1, mx1) : mx1;
        a0 = mv ? exp2f(m0 - n0) : 0.f;
        a1 = mv ? exp2f(m1 - n1) : 0.f;
      }
      const float p0 = exp2f(sc[0] - n0), p1 = exp2f(sc[1] - n1);
      const float p2 = exp2f(sc[2] - n0), p3 = exp2f(sc[3] - n1);
      l0 = l0 * a0 + p0 + p2;  // this thread's share; summed over rows at the end
      l1 = l1 * a1 + p1 + p3;
      m0 = n0;
      m1 = n1;
      mv = true;
      // running power-of-two normaliser of the V-scaled weights, raised only
      // when some lane's scale exponent passes it (else it stays, and the
      // rescale is exactly 1)
      int et = max((int)((__float_as_uint(sv0) >> 23) & 0xFF),
                   (int)((__float_as_uint(sv1) >> 23) & 0xFF));
      float rescale = 1.f;
      if (__any_sync(kFull, et > ev)) {
        et = max(et, __shfl_xor_sync(kFull, et, 4));
        et = max(et, __shfl_xor_sync(kFull, et, 8));
        et = max(et, __shfl_xor_sync(kFull, et, 16));
        const int en = min(253, max(ev, et));
        // O in units of 2^(ev-127) -> 2^(en-127): an exact power of two (or 0
        // when the old terms are below 2^-126 of the new scale)
        rescale = ev - en >= -126 ? __uint_as_float((uint32_t)(127 + ev - en) << 23) : 0.f;
        f = __uint_as_float((uint32_t)(254 - en) << 23);  // 2^(127-en)
        ev = en;
      }
      const float ra0 = a0 * rescale, ra1 = a1 * rescale;
      // O only changes scale when a running maximum moved (rare after the
      // first tiles): skip the multiplies when no column of the warp moved
      if (__any_sync(kFull, ra0 != 1.f || ra1 != 1.f)) {
#pragma unroll
        for (int kt = 0; kt < KS; ++kt) {
          o[kt][0] *= ra0; o[kt][1] *= ra1; o[kt][2] *= ra0; o[kt][3] *= ra1;
        }
        vb0 *= ra0;
        vb1 *= ra1;
      }
      const float vw0 = sv0 * f, vw1 = sv1 * f;
      sts32(p_st0, pack_f16x2(p0 * vw0, p1 * vw0));
      sts32(p_st1, pack_f16x2(p2 * vw1, p3 * vw1));
      __syncwarp();
      uint32_t pb[2];
      ldsm_x2_t(pb, pt_addr + (lane & 15) * 16);
#pragma unroll
      for (int kt = 0; kt < KS; ++kt) {
        uint32_t r0, r1, a[4];
        ldsm_b8_t(r0, r1, sVc + voff[kt]);
        i8x4_to_f16b(r0, a[0], a[2]);
        i8x4_to_f16b(r1, a[1], a[3]);
        mma_f16(o[kt], a, pb[0], pb[1]);
      }
      {
        // the bias part of the products: every A row 1152
        const uint32_t ab[4] = {kBiasF16x2, kBiasF16x2, kBiasF16x2, kBiasF16x2};
        float vb[4] = {vb0, vb1, vb0, vb1};
        mma_f16(vb, ab, pb[0], pb[1]);
        vb0 = vb[0];
        vb1 = vb[1];
      }
      __syncwarp();
    }

    if (flags & kEnd) {
      // remove the V-code bias, then back to true units: O * 2^(E-127) (0
      // when every V scale was 0 or subnormal: true terms below 2^-126)
      const float back = ev >= 1 ? __uint_as_float((uint32_t)ev << 23) : 0.f;
#pragma unroll
      for (int kt = 0; kt < KS; ++kt) {
        o[kt][0] = (o[kt][0] - vb0) * back;
        o[kt][1] = (o[kt][1] - vb1) * back;
        o[kt][2] = (o[kt][2] - vb0) * back;
        o[kt][3] = (o[kt][3] - vb1) * back;
      }
      if (!mma_segment_end<D, G>(p, pp, gph, o, m0, m1, l0, l1, mv, b, seg, flags, warp,
                                 lane, w))
        return;
    }

    __syncwarp();
    if (lane == 0) mbar_arrive(pp.empty(s));
    if (++s == pp.stages) { s = 0; ph ^= 1; }
    if (flags & kLast) break;
  }
}

// ---- fp32 consumer: CUDA-core FMAs -------------------------------------------

template <typename T, int D, int G>
struct FmaCfg {
  static constexpr int E = sizeof(T);
  static constexpr int VEC = 16 / E;    // elements per 16-byte vector
  static constexpr int EPL = D / 8;     // QK elements per lane
  static constexpr int NV = EPL / VEC;  // 16-byte vectors per lane per row
  static constexpr int PVE = D / 32;    // PV output elements per lane
  static constexpr int LOG2G = G == 1 ? 0 : G == 2 ? 1 : G == 4 ? 2 : 3;
  static constexpr int HSHIFT = 3 - LOG2G;  // after the butterfly lane i holds head i >> HSHIFT
  static_assert(NV >= 1 && PVE >= 2, "unsupported head_dim");
};

template <typename T, int D, int G>
__device__ void run_consumer_fma(const Params& p, const Pipe& pp, int warp, int lane) {
  const WaitCtl w = make_wait_ctl(p.err, p.wait_ns, p.epoch);
  using C = FmaCfg<T, D, G>;
  const int hkv = p.hkv;
  const int g = warp % hkv;
  const int wsub = warp / hkv;
  const int wph = p.nw / hkv;
  const int jg = lane >> 3;  // token slot within a pass
  const int il = lane & 7;   // lane within the token group
  const int hs = il >> C::HSHIFT;
  const bool writer = (il & ((1 << C::HSHIFT) - 1)) == 0;
  const int head_off = g * D * C::E;
  const int rs = p.rs;
  const int ST = p.st;
  float* pbuf = reinterpret_cast<float*>(pp.smem + p.off_pbuf) + warp * ST * G;
  float* mbuf = reinterpret_cast<float*>(pp.smem + p.off_mbuf);

  float qr[G][C::EPL];
  float acc[G][C::PVE];
  float m_run = -FLT_MAX, l_run = 0.f;
  bool m_valid = false;

  int s = 0;
  uint32_t ph = 0, gph = 0;
  while (true) {
    if (!mbar_wait(pp.full(s), ph, w)) return;
    const int4 d = pp.desc[s];
    const int b = d.x, n = d.y, flags = d.z, seg = d.w;
    const char* sK = reinterpret_cast<const char*>(pp.smem) + (size_t)s * pp.stage_bytes;
    const char* sV = sK + ST * rs;

    if (flags & kStart) {
      m_run = -FLT_MAX;
      m_valid = false;
      l_run = 0.f;
#pragma unroll
      for (int hh = 0; hh < G; ++hh)
#pragma unroll
        for (int e = 0; e < C::PVE; ++e) acc[hh][e] = 0.f;
      const char* qb = static_cast<const char*>(p.q) +
                       ((long long)b * p.hq + (long long)g * G) * D * C::E;
#pragma unroll
      for (int hh = 0; hh < G; ++hh)
#pragma unroll
        for (int k = 0; k < C::NV; ++k) {
          const uint4 r = ld_stream(qb + ((long long)hh * D + (il + 8 * k) * C::VEC) * C::E);
          float f[C::VEC];
          widen16<T>(r, f);
#pragma unroll
          for (int v = 0; v < C::VEC; ++v) qr[hh][k * C::VEC + v] = f[v] * p.qscale;
        }
    }

    if (n > 0) {
      float sc[kMaxPW];
#pragma unroll
      for (int pi = 0; pi < kMaxPW; ++pi) {
        const int pass = wsub + pi * wph;
        float sval = -FLT_MAX;
        bool have = false;
        if (pass * 4 < n) {
          const int t = pass * 4 + jg;
          float part[G];
#pragma unroll
          for (int hh = 0; hh < G; ++hh) part[hh] = 0.f;
          if (t < n) {
            const char* kr = sK + t * rs + head_off;
#pragma unroll
            for (int k = 0; k < C::NV; ++k) {
              const uint4 r = *reinterpret_cast<const uint4*>(kr + (il + 8 * k) * 16);
              float e[C::VEC];
              widen16<T>(r, e);
#pragma unroll
              for (int hh = 0; hh < G; ++hh)
#pragma unroll
                for (int v = 0; v < C::VEC; ++v)
                  part[hh] = fmaf(qr[hh][k * C::VEC + v], e[v], part[hh]);
            }
          }
          const float tot = butterfly<G>(part, lane);
          if (t < n) { sval = tot; have = true; }
        }
        sc[pi] = have ? sval : -INFINITY;
      }
      float mx = -INFINITY;
#pragma unroll
      for (int pi = 0; pi < kMaxPW; ++pi) mx = fmaxf(mx, sc[pi]);
      mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 16));
      float alpha = 1.f, psum = 0.f;
      if (mx != -INFINITY) {
        const float m_new = m_valid ? fmaxf(m_run, mx) : mx;
        alpha = m_valid ? exp2f(m_run - m_new) : 0.f;
#pragma unroll
        for (int pi = 0; pi < kMaxPW; ++pi) {
          const float pv = sc[pi] == -INFINITY ? 0.f : exp2f(sc[pi] - m_new);
          sc[pi] = pv;
          psum += pv;
        }
        m_run = m_new;
        m_valid = true;
      } else {
#pragma unroll
        for (int pi = 0; pi < kMaxPW; ++pi) sc[pi] = 0.f;
      }
      psum += __shfl_xor_sync(kFull, psum, 8);
      psum += __shfl_xor_sync(kFull, psum, 16);
      l_run = l_run * alpha + psum;
      if (writer) {
#pragma unroll
        for (int pi = 0; pi < kMaxPW; ++pi) {
          const int t = (wsub + pi * wph) * 4 + jg;
          if (t < n) pbuf[t * G + hs] = sc[pi];
        }
      }
      float ah[G];
#pragma unroll
      for (int hh = 0; hh < G; ++hh) ah[hh] = __shfl_sync(kFull, alpha, hh << C::HSHIFT);
      __syncwarp();
#pragma unroll
      for (int hh = 0; hh < G; ++hh)
#pragma unroll
        for (int e = 0; e < C::PVE; ++e) acc[hh][e] *= ah[hh];
      const char* vbase = sV + head_off + lane * C::PVE * C::E;
#pragma unroll
      for (int pi = 0; pi < kMaxPW; ++pi) {
        const int pass = wsub + pi * wph;
        if (pass * 4 < n) {
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const int t = pass * 4 + jj;
            if (t < n) {
              float vv[C::PVE];
              load_pv<T, C::PVE>(vbase + t * rs, vv);
              float pr[G];
#pragma unroll
              for (int hh = 0; hh < G; ++hh) pr[hh] = pbuf[t * G + hh];
#pragma unroll
              for (int hh = 0; hh < G; ++hh)
#pragma unroll
                for (int e = 0; e < C::PVE; ++e) acc[hh][e] = fmaf(pr[hh], vv[e], acc[hh][e]);
            }
          }
        }
      }
    }

    if (flags & kEnd) {
      float lh[G], mh[G];
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
        lh[hh] = __shfl_sync(kFull, l_run, hh << C::HSHIFT);
        mh[hh] = __shfl_sync(kFull, m_valid ? m_run : -INFINITY, hh << C::HSHIFT);
      }
      if (wph > 1) {
        float* mw = mbuf + warp * p.mstride;
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
#pragma unroll
          for (int e = 0; e < C::PVE; ++e) mw[hh * (D + 2) + lane * C::PVE + e] = acc[hh][e];
          if (lane == 0) { mw[hh * (D + 2) + D] = mh[hh]; mw[hh * (D + 2) + D + 1] = lh[hh]; }
        }
        if (!group_sync(pp, gph, lane, w)) return;
        if (wsub == 0) {
#pragma unroll
          for (int hh = 0; hh < G; ++hh) {
            float M = -INFINITY;
            for (int w2 = g; w2 < p.nw; w2 += hkv)
              M = fmaxf(M, mbuf[w2 * p.mstride + hh * (D + 2) + D]);
            float l = 0.f, a[C::PVE];
#pragma unroll
            for (int e = 0; e < C::PVE; ++e) a[e] = 0.f;
            if (M != -INFINITY) {
              for (int w2 = g; w2 < p.nw; w2 += hkv) {
                const float* src = mbuf + w2 * p.mstride + hh * (D + 2);
                const float mm = src[D];
                if (mm == -INFINITY) continue;
                const float wgt = exp2f(mm - M);
                l += wgt * src[D + 1];
#pragma unroll
                for (int e = 0; e < C::PVE; ++e) a[e] += wgt * src[lane * C::PVE + e];
              }
            }
            lh[hh] = l;
            mh[hh] = M;
#pragma unroll
            for (int e = 0; e < C::PVE; ++e) acc[hh][e] = a[e];
          }
        }
        if (!group_sync(pp, gph, lane, w)) return;
      }
      if (wsub == 0) {
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
          const long long row_out = (long long)b * p.hq + g * G + hh;
          const long long row_ws = (long long)seg * p.hq + g * G + hh;
          if (flags & kSingle) {
            const float inv = lh[hh] > 0.f ? 1.f / lh[hh] : 0.f;
#pragma unroll
            for (int e = 0; e < C::PVE; ++e)
              store_elem<T>(p.out, row_out * D + lane * C::PVE + e, acc[hh][e] * inv);
          } else {
            const uint64_t pol = l2_keep_policy();
#pragma unroll
            for (int e = 0; e < C::PVE; ++e)
              st_keep(p.ws_acc + row_ws * D + lane * C::PVE + e, acc[hh][e], pol);
            if (lane == 0) {
              st_keep(p.ws_ml + row_ws * 2, mh[hh], pol);
              st_keep(p.ws_ml + row_ws * 2 + 1, lh[hh], pol);
            }
          }
        }
      }
    }

    __syncwarp();
    if (lane == 0) mbar_arrive(pp.empty(s));
    if (++s == pp.stages) { s = 0; ph ^= 1; }
    if (flags & kLast) break;
  }
}

// ---- the partial-pass kernel -------------------------------------------------

template <typename T, int D, int G, int MODE>
__global__ void __launch_bounds__((consumer_warps<T>() + 1) * 32, 1)
    decode_partial_kernel(const Params p, const __grid_constant__ I8Maps maps) {
  constexpr int NW = consumer_warps<T>();
  constexpr int kThreads = (NW + 1) * 32;
  extern __shared__ __align__(1024) unsigned char smem[];
  griddep_wait();
  griddep_launch_dependents();
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;

  long long* s_cu = reinterpret_cast<long long*>(smem + p.off_cu);
  long long* s_scan = reinterpret_cast<long long*>(smem + p.off_scan);
  Pipe pp;
  pp.smem = smem;
  pp.desc = reinterpret_cast<int4*>(smem + p.off_desc);
  pp.bar0 = smem_addr(smem + p.off_bar);
  pp.stages = p.stages;
  pp.stage_bytes = p.stage_bytes;

  // ---- block counts and their exclusive scan (every CTA, same result) ----
  const int B = p.batch;
  const int per = (B + kThreads - 1) / kThreads;
  const int beg = min(B, tid * per), end = min(B, beg + per);
  const bool report = blockIdx.x == 0;
  long long local = 0;
  for (int b = beg; b < end; ++b) local += seq_blocks<MODE>(p, b, report);
  long long x = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_scan[warp] = x;
  if (tid == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(pp.full(s), 1);
      mbar_init(pp.empty(s), NW);
    }
    mbar_init(pp.group(), NW);
    mbar_init(pp.stall(), 1);
    fence_mbar_init();
  }
  __syncthreads();
  long long run = x - local;
  for (int w = 0; w < warp; ++w) run += s_scan[w];
  for (int b = beg; b < end; ++b) {
    s_cu[b] = run;
    run += seq_blocks<MODE>(p, b, false);
  }
  long long total = 0;
  for (int w = 0; w < kThreads / 32; ++w) total += s_scan[w];
  if (tid == 0) s_cu[B] = total;
  __syncthreads();

  const long long W = (total + gridDim.x - 1) / gridDim.x;
  const long long x0 = min(total, (long long)blockIdx.x * W);
  const long long x1 = min(total, x0 + W);
  if (blockIdx.x == 0) {
    const uint64_t pol = l2_keep_policy();
    for (int b = tid; b <= B; b += kThreads) st_keep(p.ws_cu + b, s_cu[b], pol);
    if (tid == 0) {
      st_keep(p.ws_meta, W, pol);
      st_keep(p.ws_meta + 1, total, pol);
    }
  }
  if (x0 >= x1) return;

  if constexpr (MODE == kModeStep) {
    // The decode step: this CTA's block range holds the last block of some
    // sequences; their new K/V rows go into the pool here, before any
    // copy of this CTA reads it.  No other CTA uses those rows: a
    // sequence's last block lies in exactly one range, and the block of a
    // new token belongs to its sequence alone (a tensor-copy box of another
    // CTA may carry them past its own rows, but those are never read).
    int b = 0, hi = B;  // first sequence ending at or after block x0
    while (b < hi) {
      const int mid = (b + hi) >> 1;
      if (s_cu[mid + 1] - 1 < x0) b = mid + 1; else hi = mid;
    }
    const int pieces = p.row_bytes / 16;
    for (; b < B && s_cu[b + 1] - 1 < x1; ++b) {
      if (s_cu[b + 1] == s_cu[b]) continue;  // empty (or refused) sequence
      const long long pos = (long long)(p.offs ? p.offs[b] : 0) + p.lens[b] - 1;
      const int blk = p.bt[(long long)b * p.mb + pos / p.bs];
      if (blk < 0 || (long long)blk >= p.num_blocks) continue;  // the producer reports it
      const long long dst = (long long)blk * p.block_stride + (pos % p.bs) * p.row_bytes;
      const long long src = (long long)b * p.new_row_bytes;
      if constexpr (sizeof(T) == 1) {
        // int8 pool: warp g quantises kv head g of the new K and V rows,
        // exactly as the quantising scatter does
        constexpr int VPL = D / 32;
        if (warp < p.hkv) {
          const long long e = src + ((long long)warp * D + lane * VPL) * 2;
          float xk[VPL], xv[VPL];
          load_bf16<VPL>(reinterpret_cast<const __nv_bfloat16*>(p.k_new + e), xk);
          load_bf16<VPL>(reinterpret_cast<const __nv_bfloat16*>(p.v_new + e), xv);
          int ck[VPL], cv[VPL];
          const float sk = quantise_head<VPL>(xk, ck);
          const float sv = quantise_head<VPL>(xv, cv);
          store_codes<VPL>(p.k_out + dst + warp * D + lane * VPL, ck);
          store_codes<VPL>(p.v_out + dst + warp * D + lane * VPL, cv);
          if (lane == 0) {
            *reinterpret_cast<float*>(p.k_out + dst + p.scale_off + 4 * warp) = sk;
            *reinterpret_cast<float*>(p.v_out + dst + p.scale_off + 4 * warp) = sv;
          }
        }
      } else {
        for (int i = tid; i < 2 * pieces; i += kThreads) {
          const bool vh = i >= pieces;
          const long long o = 16ll * (vh ? i - pieces : i);
          const uint4 x = *reinterpret_cast<const uint4*>((vh ? p.v_new : p.k_new) + src + o);
          *reinterpret_cast<uint4*>((vh ? p.v_out : p.k_out) + dst + o) = x;
        }
      }
    }
    // the rows just stored are read next by the copies (async proxy)
    fence_proxy_async_global();
    __syncthreads();
  }

  if (warp == NW) {
    run_producer<sizeof(T) == 1 ? kStageI8 : sizeof(T) == 2 ? kStageBf16 : kStageRows, MODE>(
        p, pp, maps, s_cu, lane, x0, x1);
    return;
  }
  if (p.skip_fill == 2 || (p.skip_fill == 1 && blockIdx.x == 0)) {
    // test hook: the consumers first wait on a barrier nothing arrives at,
    // which can only give up at the bound; they then leave without
    // releasing a stage, so the producer's wait for a free stage gives up too
    mbar_wait(pp.stall(), 0, make_wait_ctl(p.err, p.wait_ns, p.epoch));
    return;
  }
  if constexpr (sizeof(T) == 1) {
    run_consumer_i8<D, G>(p, pp, warp, lane);
  } else if constexpr (sizeof(T) == 2) {
    run_consumer_mma<D, G>(p, pp, warp, lane);
  } else {
    run_consumer_fma<T, D, G>(p, pp, warp, lane);
  }
}

// Merge the partial states of every segment of a sequence.  One warp per
// (sequence, q head); lane i holds the D/32 consecutive outputs d = i D/32 ..
// The segments are the shared-prefix states (nsplit of them, prefix pass of
// shared-prefix decode; none otherwise) followed by the sequence's segments
// of the partial pass.  The lanes load 32 segments' (m, l) at once, take
// their maximum and weights by warp reductions, then every lane adds the
// weighted accumulators of those segments with independent vector loads:
// two dependent memory round trips per 32 segments, and one wave of warps
// for the batch.  Sequences the partial pass finished itself (wholly inside
// one CTA, no prefix states) are skipped; a sequence with no tokens gets
// zeros.  The loads are evict-first: the states are dead once read.
template <typename T, int D>
__global__ void __launch_bounds__(256)
    decode_combine_kernel(const float* __restrict__ ws_acc, const float* __restrict__ ws_ml,
                          const long long* __restrict__ ws_cu,
                          const long long* __restrict__ ws_meta,
                          const float* __restrict__ pre_acc, const float* __restrict__ pre_ml,
                          int nsplit, int batch, int hq, T* __restrict__ out) {
  constexpr int VPL = D / 32;
  griddep_wait();
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const long long wid = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (wid >= (long long)batch * hq) return;
  const int b = (int)(wid / hq), h = (int)(wid - (long long)b * hq);
  T* o = out + wid * D + lane * VPL;
  // the three index words in one round trip
  const long long c0 = __ldcs(ws_cu + b), c1 = __ldcs(ws_cu + b + 1);
  const long long W = __ldcs(ws_meta);
  long long cf = 0, nsuf = 0;
  if (c1 > c0) {
    cf = c0 / W;
    nsuf = (c1 - 1) / W - cf + 1;
  }
  if (nsplit == 0 && nsuf <= 1) {
    if (nsuf == 0) {  // no tokens (or an invalid sequence): zeros
#pragma unroll
      for (int e = 0; e < VPL; ++e) o[e] = T(0.f);
    }
    return;
  }
  const long long nseg = nsplit + nsuf;
  // state row of segment sg: a prefix state, or a partial-pass segment
  auto row_of = [&](long long sg) -> long long {
    return sg < nsplit ? ((long long)sg * batch + b) * hq + h : (cf + (sg - nsplit) + b) * hq + h;
  };
  auto load_acc = [&](long long sg, float (&v)[VPL]) {
    const float* a = (sg < nsplit ? pre_acc : ws_acc) + row_of(sg) * D + lane * VPL;
    if constexpr (VPL == 4) {
      const float4 x = __ldcs(reinterpret_cast<const float4*>(a));
      v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
    } else {
      const float2 x = __ldcs(reinterpret_cast<const float2*>(a));
      v[0] = x.x; v[1] = x.y;
    }
  };
  constexpr int kAhead = 4;  // accumulators loaded together with the chunk's (m, l)
  float M = -INFINITY, den = 0.f, acc[VPL];
#pragma unroll
  for (int e = 0; e < VPL; ++e) acc[e] = 0.f;
  for (long long base = 0; base < nseg; base += 32) {
    const int n = (int)min(32ll, nseg - base);
    const long long sl = base + lane;
    float m = -INFINITY, l = 0.f;
    if (sl < nseg) {
      const float2 v =
          __ldcs(reinterpret_cast<const float2*>((sl < nsplit ? pre_ml : ws_ml) + 2 * row_of(sl)));
      m = v.x;
      l = v.y;
    }
    // the first accumulators of the chunk, in flight with the (m, l) loads
    float av[kAhead][VPL];
#pragma unroll
    for (int j = 0; j < kAhead; ++j) {
      if (j < n) load_acc(base + j, av[j]);
      else
#pragma unroll
        for (int e = 0; e < VPL; ++e) av[j][e] = 0.f;
    }
    float cm = m;
#pragma unroll
    for (int x = 16; x > 0; x >>= 1) cm = fmaxf(cm, __shfl_xor_sync(kFull, cm, x));
    if (cm == -INFINITY) continue;  // no keys in these segments
    const float nM = fmaxf(M, cm);
    const float r = exp2f(M - nM);  // 0 while M is still -inf (the sums are 0 then)
    den *= r;
#pragma unroll
    for (int e = 0; e < VPL; ++e) acc[e] *= r;
    M = nM;
    const float wgt = m == -INFINITY ? 0.f : exp2f(m - nM);
    float wl = wgt * l;
#pragma unroll
    for (int x = 16; x > 0; x >>= 1) wl += __shfl_xor_sync(kFull, wl, x);
    den += wl;
#pragma unroll
    for (int j = 0; j < kAhead; ++j) {
      const float wj = __shfl_sync(kFull, wgt, j);  // 0 past n: no segment
#pragma unroll
      for (int e = 0; e < VPL; ++e) acc[e] += wj * av[j][e];
    }
#pragma unroll 4
    for (int j = kAhead; j < n; ++j) {
      const float wj = __shfl_sync(kFull, wgt, j);
      float v[VPL];
      load_acc(base + j, v);
#pragma unroll
      for (int e = 0; e < VPL; ++e) acc[e] += wj * v[e];
    }
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
#pragma unroll
  for (int e = 0; e < VPL; ++e) o[e] = T(acc[e] * inv);
}

// ---- host side -----------------------------------------------------------------

int stage_tokens(int bs, int row_bytes) {
  int st = 1;
  while (st * 2 <= kMaxStageTokens && st * 2 <= bs && st * 2 * row_bytes <= 32768) st *= 2;
  return st;
}

struct Layout {
  int st, rs, vrs, stages, smem, off_bar, off_desc, off_cu, off_scan, off_pbuf, off_mbuf,
      off_vbuf;
  int stage_bytes, off_kc, off_vc, off_ks, off_vs, tx_bytes, sbytes;  // see Params
  int box_rows, box_bytes, halves;                                    // see Params
};

int align_up(int x, int a) { return (x + a - 1) / a * a; }

Layout make_layout(int bs, int row_bytes, int hkv, int G, int D, int batch, int smem_optin,
                   bool quant, bool elem2, int nw) {
  Layout L{};
  L.st = stage_tokens(bs, row_bytes);
  L.rs = row_bytes + kRowPad;
  L.vrs = 0;
  const int vbuf = 0;
  if (quant) {
    // [K codes (Hkv, st, D) | V codes | K scales (st, sbytes) | V scales]:
    // every tensor-copy destination 128-byte aligned, the swizzled code
    // tiles 1024-byte aligned
    const int codes = hkv * L.st * D;
    L.sbytes = (4 * hkv + 15) / 16 * 16;
    L.off_kc = 0;
    L.off_vc = align_up(codes, 1024);
    L.off_ks = 2 * align_up(codes, 1024);
    L.off_vs = align_up(L.off_ks + L.st * L.sbytes, 128);
    L.stage_bytes = align_up(L.off_vs + L.st * L.sbytes, 1024);
    L.tx_bytes = 2 * codes + 2 * L.st * L.sbytes;
  } else if (elem2) {
    // bf16: per stage, tensor-copy boxes of (64 elements, box_rows rows,
    // Hkv heads) with the 128-byte swizzle, K halves then V halves; a box
    // holds Hkv * box_rows lines of 128 bytes, at least 8 so that every box
    // is a whole number of 1024-byte swizzle blocks
    L.halves = D / 64;
    L.box_rows = L.st;
    while (hkv * L.box_rows < 8) L.box_rows *= 2;
    L.box_bytes = hkv * L.box_rows * 128;
    L.stage_bytes = 2 * L.halves * L.box_bytes;
    L.tx_bytes = L.stage_bytes;
  } else {
    L.stage_bytes = 2 * L.st * L.rs;
  }
  const int stage_bytes = L.stage_bytes;
  const int pbuf = nw * (quant ? 256 : (L.st * G * 4 > 256 ? L.st * G * 4 : 256));
  // merge buffers of warps sharing a kv head
  const int mbuf = hkv < nw ? 4 * nw * G * (D + 2) : 0;
  int fixed = 0;
  fixed += 8 * (2 * kMaxStages + 2);              // barriers
  fixed = align_up(fixed, 16) + 16 * kMaxStages;  // descriptors
  fixed = align_up(fixed, 16) + 8 * (batch + 1);  // cu
  fixed = align_up(fixed, 16) + 8 * 32;           // scan scratch
  fixed = align_up(fixed, 16) + pbuf;
  fixed = align_up(fixed, 16) + mbuf;
  fixed = align_up(fixed, 16) + vbuf;
  fixed = align_up(fixed, 128);
  if (quant && (L.off_vc % 1024 || L.off_ks % 128 || L.off_vs % 128 || stage_bytes % 1024))
    return L;  // stages 0: refused (every tensor copy needs an aligned destination)
  if (elem2 && (L.box_bytes % 1024 || (D != 64 && D != 128))) return L;  // the same
  int stages = (smem_optin - fixed) / stage_bytes;
  if (stages > kMaxStages) stages = kMaxStages;
  L.stages = stages;
  int off = align_up(stages * stage_bytes, 128);
  L.off_bar = off;   off += 8 * (2 * stages + 2);
  off = align_up(off, 16); L.off_desc = off; off += 16 * stages;
  off = align_up(off, 16); L.off_cu = off;   off += 8 * (batch + 1);
  off = align_up(off, 16); L.off_scan = off; off += 8 * 32;
  off = align_up(off, 16); L.off_pbuf = off; off += pbuf;
  off = align_up(off, 16); L.off_mbuf = off; off += mbuf;
  off = align_up(off, 16); L.off_vbuf = off; off += vbuf;
  L.smem = align_up(off, 16);
  return L;
}

// Workspace carve (bytes): meta [W, total] | cu[batch+1] (int64) |
// (m, l) per (segment, q head) | acc per (segment, q head, d); segments are
// indexed c + b, so grid + batch of them suffice.
struct WsLayout {
  size_t meta, cu, ml, acc, total;
};

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

WsLayout ws_layout(int batch, int hq, int D, int grid) {
  WsLayout w{};
  const size_t parts = (size_t)grid + (size_t)batch;
  w.meta = 0;
  w.cu = 256;
  w.ml = w.cu + round256(8 * ((size_t)batch + 1));
  w.acc = w.ml + round256(parts * hq * 2 * 4);
  w.total = w.acc + round256(parts * hq * D * 4);
  return w;
}

// Dynamic shared memory, configured once per kernel instance and device
// (`configured` is the caller's per-instance cache).
template <typename K>
cudaError_t ensure_smem(K kern, int smem, int (&configured)[64]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && configured[dev] >= smem) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess && dev >= 0 && dev < 64) configured[dev] = smem;
  return e;
}

template <typename T, int D, int G, int MODE>
cudaError_t run(const DecodeLaunch& a, const Layout& L, cudaStream_t s) {
  const PoolView& pv = a.pool;
  Params p{};
  const long long layer_off = (long long)a.layer * pv.block_size * pv.row_bytes;
  p.k_base = pv.k + layer_off;
  p.v_base = pv.v + layer_off;
  p.block_stride = (long long)pv.num_layers * pv.block_size * pv.row_bytes;
  p.num_blocks = pv.num_blocks;
  p.q = a.q;
  p.out = a.out;
  p.bt = a.bt;
  p.lens = a.lens;
  p.offs = a.offs;
  const int grid = a.grid;
  const WsLayout W = ws_layout(a.batch, a.num_q_heads, pv.head_dim, grid);
  char* ws = static_cast<char*>(a.workspace);
  p.ws_meta = reinterpret_cast<long long*>(ws + W.meta);
  p.ws_cu = reinterpret_cast<long long*>(ws + W.cu);
  p.ws_ml = reinterpret_cast<float*>(ws + W.ml);
  p.ws_acc = reinterpret_cast<float*>(ws + W.acc);
  p.err = a.err;
  p.mb = a.mb;
  p.batch = a.batch;
  p.hq = a.num_q_heads;
  p.hkv = pv.num_kv_heads;
  p.bs = pv.block_size;
  p.row_bytes = pv.row_bytes;
  p.rs = L.rs;
  p.st = L.st;
  p.stages = L.stages;
  p.vrs = L.vrs;
  p.stage_bytes = L.stage_bytes;
  p.nw = consumer_warps<T>();
  p.mstride = G * (D + 2);
  p.off_kc = L.off_kc;
  p.off_vc = L.off_vc;
  p.off_ks = L.off_ks;
  p.off_vs = L.off_vs;
  p.tx_bytes = L.tx_bytes;
  p.sbytes = L.sbytes;
  p.box_rows = L.box_rows;
  p.box_bytes = L.box_bytes;
  p.halves = L.halves;
  p.rows_per_block = (long long)pv.num_layers * pv.block_size;
  p.layer_row = a.layer * pv.block_size;
  p.qscale = a.scale * kLog2e;
  p.off_bar = L.off_bar;
  p.off_desc = L.off_desc;
  p.off_cu = L.off_cu;
  p.off_scan = L.off_scan;
  p.off_pbuf = L.off_pbuf;
  p.off_mbuf = L.off_mbuf;
  p.off_vbuf = L.off_vbuf;
  p.k_new = a.k_new;
  p.v_new = a.v_new;
  p.k_out = pv.k_mut ? pv.k_mut + layer_off : nullptr;
  p.v_out = pv.v_mut ? pv.v_mut + layer_off : nullptr;
  p.new_row_bytes = pv.num_kv_heads * pv.head_dim * pv.io_size;
  p.scale_off = pv.scale_off;
  p.prefix_blocks = a.prefix_blocks;
  p.wait_ns = wait_limit_ns();
  p.epoch = next_launch_epoch();
  p.skip_fill = debug_skip_fill();

  I8Maps maps;
  memset(&maps, 0, sizeof(maps));
  if constexpr (sizeof(T) == 1) {
    const int H = pv.num_kv_heads;
    const cuuint64_t rows = (cuuint64_t)pv.num_blocks * pv.num_layers * pv.block_size;
    const cuuint64_t cdims[3] = {(cuuint64_t)D, rows, (cuuint64_t)H};
    const cuuint64_t cstrides[2] = {(cuuint64_t)pv.row_bytes, (cuuint64_t)D};
    const cuuint32_t cbox[3] = {(cuuint32_t)D, (cuuint32_t)L.st, (cuuint32_t)H};
    const CUtensorMapSwizzle sw = D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    const cuuint64_t sdims[2] = {(cuuint64_t)L.sbytes, rows};
    const cuuint64_t sstrides[1] = {(cuuint64_t)pv.row_bytes};
    const cuuint32_t sbox[2] = {(cuuint32_t)L.sbytes, (cuuint32_t)L.st};
    if (!encode_tiled(&maps.kc, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, pv.k, cdims, cstrides, cbox, sw) ||
        !encode_tiled(&maps.vc, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, pv.v, cdims, cstrides, cbox, sw) ||
        !encode_tiled(&maps.ks, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, pv.k + pv.scale_off, sdims,
                      sstrides, sbox, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_tiled(&maps.vs, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, pv.v + pv.scale_off, sdims,
                      sstrides, sbox, CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
  }
  if constexpr (sizeof(T) == 2) {
    // bf16: K and V as (d, token row, kv head) boxes of (64, box_rows, Hkv)
    // elements with the 128-byte swizzle
    const cuuint64_t rows = (cuuint64_t)pv.num_blocks * pv.num_layers * pv.block_size;
    const cuuint64_t dims[3] = {(cuuint64_t)D, rows, (cuuint64_t)pv.num_kv_heads};
    const cuuint64_t strides[2] = {(cuuint64_t)pv.row_bytes, (cuuint64_t)D * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)L.box_rows, (cuuint32_t)pv.num_kv_heads};
    if (!encode_tiled(&maps.kc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, pv.k, dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tiled(&maps.vc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, pv.v, dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  auto kern = decode_partial_kernel<T, D, G, MODE>;
  static int configured[64] = {0};
  cudaError_t e = ensure_smem(kern, L.smem, configured);
  if (e != cudaSuccess) return e;
  // programmatic dependent launches, except when the caller times the partial
  // pass alone with events (an event between kernels ends the overlap)
  const bool pdl = a.ev_start == nullptr && a.ev_stop == nullptr;
  if (a.ev_start && (e = cudaEventRecord(a.ev_start, s)) != cudaSuccess) return e;
  e = launch_kernel(kern, dim3(grid), dim3((consumer_warps<T>() + 1) * 32), L.smem, s, pdl, p,
                    maps);
  if (e != cudaSuccess) return e;
  if (a.ev_stop && (e = cudaEventRecord(a.ev_stop, s)) != cudaSuccess) return e;
  // the suffix pass of shared-prefix decode: its combine runs after the
  // prefix pass (launch_decode_combine_prefix)
  if constexpr (MODE == kModeSuffix) return cudaSuccess;
  // int8 pools take and return bf16
  using OutT = std::conditional_t<sizeof(T) == 1, __nv_bfloat16, T>;
  const unsigned cgrid = (unsigned)(((long long)a.batch * p.hq + 7) / 8);
  return launch_kernel(decode_combine_kernel<OutT, D>, dim3(cgrid), dim3(256), 0, s, pdl,
                       (const float*)p.ws_acc, (const float*)p.ws_ml, (const long long*)p.ws_cu,
                       (const long long*)p.ws_meta, (const float*)nullptr, (const float*)nullptr,
                       0, a.batch, p.hq, static_cast<OutT*>(a.out));
}

template <typename T, int D, int MODE>
cudaError_t run_gf(const DecodeLaunch& a, const Layout& L, int G, cudaStream_t s) {
  switch (G) {
    case 1: return run<T, D, 1, MODE>(a, L, s);
    case 2: return run<T, D, 2, MODE>(a, L, s);
    case 4: return run<T, D, 4, MODE>(a, L, s);
    case 8: return run<T, D, 8, MODE>(a, L, s);
  }
  return cudaErrorInvalidValue;
}

template <typename T, int D>
cudaError_t run_g(const DecodeLaunch& a, const Layout& L, int G, cudaStream_t s) {
  if (a.prefix_blocks > 0) {
    // the suffix pass exists for the shapes the prefix pass supports
    if constexpr (std::is_same_v<T, __nv_bfloat16> && D == 128)
      return run_gf<T, D, kModeSuffix>(a, L, G, s);
    return cudaErrorInvalidConfiguration;
  }
  return a.k_new ? run_gf<T, D, kModeStep>(a, L, G, s) : run_gf<T, D, kModePlain>(a, L, G, s);
}

}  // namespace

size_t decode_workspace_bytes(int batch, int num_q_heads, int head_dim, int grid) {
  const int bmax = batch < kDecodeMaxBatch ? batch : kDecodeMaxBatch;
  return ws_layout(bmax > 0 ? bmax : 0, num_q_heads, head_dim, grid).total;
}

int decode_supported(const PoolView& p, int num_q_heads) {
  if (p.head_dim != 64 && p.head_dim != 128) return 1;
  const int hkv = p.num_kv_heads;
  if (hkv != 1 && hkv != 2 && hkv != 4 && hkv != 8) return 1;
  if (num_q_heads % hkv) return 1;
  const int G = num_q_heads / hkv;
  if (G != 1 && G != 2 && G != 4 && G != 8) return 1;
  return 0;
}

cudaError_t launch_decode(const DecodeLaunch& a, cudaStream_t s) {
  const PoolView& pv = a.pool;
  const int G = a.num_q_heads / pv.num_kv_heads;
  const Layout L = make_layout(pv.block_size, pv.row_bytes, pv.num_kv_heads, G, pv.head_dim,
                               a.batch, a.smem_optin, pv.quant != 0,
                               pv.quant == 0 && pv.elem_size == 2, pv.quant ? kNWI8 : kNW);
  if (L.stages < 2) return cudaErrorInvalidConfiguration;
  if (pv.quant) {
    // tensor-copy row coordinates are 32-bit
    if ((long long)pv.num_blocks * pv.num_layers * pv.block_size >= (1ll << 31))
      return cudaErrorInvalidConfiguration;
    return pv.head_dim == 128 ? run_g<int8_t, 128>(a, L, G, s) : run_g<int8_t, 64>(a, L, G, s);
  }
  if (pv.elem_size == 2) {
    // tensor-copy row coordinates are 32-bit
    if ((long long)pv.num_blocks * pv.num_layers * pv.block_size >= (1ll << 31))
      return cudaErrorInvalidConfiguration;
    return pv.head_dim == 128 ? run_g<__nv_bfloat16, 128>(a, L, G, s)
                              : run_g<__nv_bfloat16, 64>(a, L, G, s);
  }
  return pv.head_dim == 128 ? run_g<float, 128>(a, L, G, s) : run_g<float, 64>(a, L, G, s);
}

cudaError_t launch_decode_combine_prefix(const DecodeLaunch& a, const float* pre_ml,
                                         const float* pre_acc, int nsplit, cudaStream_t s) {
  const int D = a.pool.head_dim;
  const WsLayout W = ws_layout(a.batch, a.num_q_heads, D, a.grid);
  const char* ws = static_cast<const char*>(a.workspace);
  if (D != 128) return cudaErrorInvalidValue;
  const unsigned cgrid = (unsigned)(((long long)a.batch * a.num_q_heads + 7) / 8);
  return launch_kernel(decode_combine_kernel<__nv_bfloat16, 128>, dim3(cgrid), dim3(256), 0, s,
                       true, reinterpret_cast<const float*>(ws + W.acc),
                       reinterpret_cast<const float*>(ws + W.ml),
                       reinterpret_cast<const long long*>(ws + W.cu),
                       reinterpret_cast<const long long*>(ws + W.meta), pre_acc, pre_ml, nsplit,
                       a.batch, a.num_q_heads, static_cast<__nv_bfloat16*>(a.out));
}

}  // namespace pkv
