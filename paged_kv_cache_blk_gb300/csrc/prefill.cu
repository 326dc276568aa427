// Paged prefill attention on the 5th-generation tensor cores (tcgen05, TMEM,
// TMA).
//
// What is computed (the prefill batch of "vLLM PagedAttention source notes"
// §2.4: every prompt token's K/V is computed and written into its blocks, then
// attention runs over them): the last n_b tokens of sequence b are queries;
// query i sits at logical position P_i = seq_len_b - n_b + i and attends
// causally to the keys 0..P_i of the sequence, read in place from the pool
// through the block table (first-block offset honoured).  GQA: query head h
// reads kv head h / (Hq / Hkv).
//
// Work items are (pair of query tiles, sequence, kv head), taken in turn by a
// persistent grid of one CTA per SM; for prefill the CTAs run in pairs (two-
// CTA clusters) that share every K/V tile (below):
//  * A query tile is 128 MMA rows = (128 / G) query tokens x the G query
//    heads of kv head g, so each K/V tile feeds all G heads (row r = token *
//    G + head).  The CTA owns two tiles, A and B, that share the K/V stream.
//  * Keys in tiles of 128 table positions (128 / bs whole blocks).  K(t) and
//    V(t) are loaded by TMA (one box per block and 64-column half, 128B
//    swizzle) into a 4-slot ring in the order K0 V0 K1 V1 ...; invalid table
//    entries load zeros.
//  * Warp 9 issues S_x = Q_x K^T (M 128, N 128, K 128: 8 tcgen05.mma, fp32
//    in TMEM) and O_x += P_x V (V is the MN-major operand) in the order
//    S_A(0) S_B(0) | PV_A(t) S_A(t+1) PV_B(t) S_B(t+1) | ..., so the softmax
//    of one tile runs while the tensor cores work on the other.  Its thread
//    advances in step with the tensor cores (their queue holds about one
//    instruction), so it does little else: the item values come from the
//    loads warp (warp 8) through a small shared-memory ring.
//  * Warps 0-3 (tile A) and 4-7 (tile B) own one row each: they read the S
//    row from TMEM (tcgen05.ld 32x32b), mask only the tiles and 32-key
//    chunks that need it (a chunk masked for every row of the warp gets P = 0
//    without exponentials), keep
//    the running sum and a maximum that moves only when a score exceeds it by
//    more than 8 in log2 units (checked per 32-key chunk before that chunk's
//    P is stored; the O row is then rescaled in TMEM), and write P as bf16
//    pairs over the S columns in TMEM, the A operand of the second MMA.
//  * Epilogue: O row / l -> bf16 -> global (only rows that are real queries).
//  * CTA pairs: the two CTAs of a cluster take neighbouring tile pairs of one
//    (sequence, kv head), so they stream the same K/V tiles.  Each loads one
//    64-column half of every tile by TMA and copies it into the other CTA's
//    ring (a shared-memory bulk copy within the cluster), so each tile is
//    read from L2 once for both SMs.  No tensor copy is multicast.
// Every wait is bounded; on a timeout the CTA records the error, drains its
// MMAs and frees its TMEM before returning.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

#include "common.cuh"
#include "pkv.h"
#include "tma.cuh"

namespace pkv {
namespace {

constexpr int kPfWarps = 10;  // 0-3 softmax A, 4-7 softmax B, 8 TMA, 9 MMA
constexpr int kWarpTma = 8;
constexpr int kWarpMma = 9;
constexpr int kWarpFwd = 10;  // CTA pairs: forwards this CTA's halves to the other CTA
// threads of a CTA: one more warp in a CTA pair
template <bool SHARE>
constexpr int pf_threads() {
  return (kPfWarps + (SHARE ? 1 : 0)) * 32;
}
constexpr int kRows = 128;   // MMA M: query rows per tile
constexpr int kKeys = 128;   // keys per KV tile (MMA N of Q K^T, K of P V)
constexpr int kD = 128;      // head_dim
constexpr int kHalf = 128 * 64 * 2;  // one 128-row x 64-column bf16 half tile (16 KB)
constexpr int kTileBytes = 2 * kHalf;  // 32 KB
constexpr int kSlots = 4;              // K / V ring: K(t) V(t) K(t+1) V(t+1)
constexpr uint32_t kTmemCols = 512;    // S_A, S_B, O_A, O_B
constexpr float kLog2e = 1.4426950408889634f;

// shared-memory carve, from a 1024-aligned base
constexpr int kOffQ = 0;                              // Q_A, Q_B
constexpr int kOffKV = 2 * kTileBytes;                // ring of kSlots tiles
constexpr int kOffBar = kOffKV + kSlots * kTileBytes;
constexpr int kOffTslot = kOffBar + 320;              // TMEM address, after the barriers
constexpr int kItemRing = 4;                          // items the loads warp publishes ahead
constexpr int kOffItems = kOffBar + 512;              // [kItemRing][own item, lead item]
constexpr int kSmemBytes = kOffItems + 1024 + 1024;   // + alignment slack

struct PfParams {
  const int32_t* bt;
  const int32_t* lens;
  const int32_t* offs;
  const long long* cu_q;
  void* out;
  int* err;
  long long total_q;
  long long blk_coord_limit;  // N * L (coordinate of the combined block/layer dimension)
  long long num_blocks;
  long long n_items;  // pairs x batch x kv heads
  int mb, batch, hq, hkv, G, TQ, bs, L, layer, max_q_len;
  float qscale;
  // shared-prefix decode (prefix pass): the queries are the decode queries of
  // the batch's sequences (q [batch, hq, D]); the keys are the first
  // prefix_blocks entries of table row 0, in key_tiles tiles split into
  // nsplit ranges of per_split tiles; the states go to pre_ml / pre_acc
  int prefix_blocks, key_tiles, nsplit, per_split;
  float* pre_ml;
  float* pre_acc;
  unsigned long long wait_ns;  // bound of one wait (0 = the default)
  int epoch;  // this launch's number (see WaitCtl)
  int skip_fill;  // test hook: 1 = CTA 0, 2 = every CTA stalls its MMA warp
};

// ---- tcgen05 / TMA helpers ----------------------------------------------------

__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFF);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= 1ull << 46;  // descriptor version for this architecture
  d |= 2ull << 61;  // 128-byte swizzle
  return d;
}

// kind::f16 instruction descriptor: fp32 accumulate, bf16 A and B, M 128, N 128.
constexpr uint32_t kIdescKK =
    (1u << 4) | (1u << 7) | (1u << 10) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
constexpr uint32_t kIdescKMN = kIdescKK | (1u << 16);  // B MN-major

__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                     uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The same with the A operand in TMEM (M rows = lanes; column c holds the
// bf16 pair of k = 2c (low half) and 2c + 1; a K = 16 step spans 8 columns).
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// The same arrive on the barrier at address `bar` in both CTAs of a pair (an
// arrive signal only: no data moves between the CTAs).
__device__ __forceinline__ void umma_commit_both(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"((uint16_t)3)
      : "memory");
}

// ---- CTA pairs (clusters of two that share their K/V tiles) -------------------------

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// shared::cluster address of this CTA's shared address `a` in CTA `rank`
__device__ __forceinline__ uint32_t peer_addr(uint32_t a, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  return r;
}

// arrive on a barrier of the other CTA of the pair (cluster address)
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// bytes of this CTA's shared memory at `src` to `dst` in the other CTA's
// (cluster address), completion counted as transaction bytes on that CTA's
// barrier `bar` (cluster address); 16-byte aligned, a multiple of 16 bytes
__device__ __forceinline__ void bulk_s2s(uint32_t dst, uint32_t src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, "
      "[%3];" ::"r"(dst),
      "r"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// every thread of both CTAs
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::
          : "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
        "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
      "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
      "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---- the kernel ------------------------------------------------------------------

// Rows of the S / P tile per thread of a softmax warpgroup (one row per
// thread), and the state a warpgroup keeps for its query tile.
struct RowState {
  float m_used;  // the maximum P is taken against (raised only by more than 8)
  float l;       // running sum of P
};

__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Softmax of one S tile for one row: reads the row from TMEM, masks it,
// updates the running state, rescales the O row when the maximum moved, and
// writes the row's P as bf16 pairs back into TMEM, where the P V product reads
// it as its A operand.
__device__ __forceinline__ void softmax_tile(uint32_t tS, uint32_t tO, uint32_t lane_base, int t,
                                             int c_lo, int c_hi, bool full_tile, float qs,
                                             RowState& st) {
  // With a positive scale the maximum is taken on the raw scores and the scale
  // goes into the exponent's FMA; otherwise each score is scaled first.
  const bool pre = qs <= 0.f;
  const float qe = pre ? 1.f : qs;
  // one 32-column chunk of the S row, scaled when needed and masked (the key
  // in column c is valid for c_lo <= c <= c_hi)
  auto load_chunk = [&](int c0, float (&x)[32]) {
    uint32_t v[32];
    tmem_ld32(tS + lane_base + c0, v);
    tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      float f = __uint_as_float(v[j]);
      if (pre) f *= qs;
      if (!full_tile) f = (c0 + j >= c_lo && c0 + j <= c_hi) ? f : -INFINITY;
      x[j] = f;
    }
  };
  // P of one chunk against the maximum mu as bf16 pairs, and their sum (a row
  // with no maximum yet uses 0; a finite score then raises it and this P is
  // recomputed)
  auto p_chunk = [&](const float (&x)[32], float mu, uint32_t (&w)[16]) {
    float psum = 0.f;
    const float ms = mu == -INFINITY ? 0.f : mu;
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const float y0 = fmaf(x[2 * e], qe, -ms), y1 = fmaf(x[2 * e + 1], qe, -ms);
      const float a0 = exp2f(y0), a1 = exp2f(y1);
      psum += a0 + a1;
      w[e] = pack_bf16x2(a0, a1);
    }
    return psum;
  };
  // maximum of a chunk as four independent chains, so its latency is short
  auto chunk_max = [&](const float (&x)[32]) {
    float m[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float* y = x + 8 * k;
      m[k] = fmaxf(max3(max3(max3(y[0], y[1], y[2]), y[3], y[4]), y[5], y[6]), y[7]);
    }
    return fmaxf(max3(m[0], m[1], m[2]), m[3]);
  };
  // P (bf16 pairs) of chunk c0 goes to TMEM columns c0/2 .. c0/2 + 15 of the S
  // region, the A operand of O += P V.  Those columns hold S values of this
  // chunk or of earlier ones, all read before.
  //
  // Every tcgen05.ld / st below is a warp-wide instruction, so all control
  // flow around them is warp-uniform: per-row decisions only select data.
  // The O rescale needs P(t-1) V(t-1) to have completed; it has, because
  // S(t) was issued after it and its commit (the "S ready" barrier) covers
  // every earlier product.
  float psum = 0.f, alpha = 1.f;
  {
    // One pass against the maximum in use.  Each chunk's maximum is checked
    // before its P is kept: a row whose chunk maximum lies more than 8 above
    // the maximum in use raises it to that chunk maximum, scales the P it
    // stored for earlier chunks (bf16, in place) and their sum by
    // 2^(old - new), and recomputes the chunk's P.  So no stored P exceeds
    // 2^8 and no exponential overflows, however far a later score jumps.  A
    // row with no maximum yet (-inf: its first tile) takes the first chunk
    // holding one of its keys as its maximum the same way (its earlier P are
    // zeros); a padding row, all keys masked, keeps P = 0 throughout.
    float mu = st.m_used;
#pragma unroll 1
    for (int c0 = 0; c0 < kKeys; c0 += 32) {
      float x[32];
      // in a masked tile (the causal diagonal) a chunk is often outside every
      // row's keys of the warp (its P is zero: no exponentials) or inside all
      // of them (no mask code); the votes keep the TMEM accesses warp-uniform
      bool plain = full_tile;
      if (!full_tile) {
        if (__all_sync(0xffffffffu, c0 > c_hi || c0 + 31 < c_lo)) {
          const uint32_t z[16] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u,
                                  0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
          tmem_st16(tS + lane_base + (c0 >> 1), z);
          continue;
        }
        plain = __all_sync(0xffffffffu, c0 >= c_lo && c0 + 31 <= c_hi);
      }
      if (plain && !pre) {
        // the common case, kept free of masking and scaling code
        uint32_t v[32];
        tmem_ld32(tS + lane_base + c0, v);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(v[j]);
      } else {
        load_chunk(c0, x);
      }
      const float cm = chunk_max(x) * qe;
      uint32_t w[16];
      float ps = p_chunk(x, mu, w);
      // stored before the check so the store does not wait for the maximum;
      // a row that raises its maximum overwrites it below
      tmem_st16(tS + lane_base + (c0 >> 1), w);
      if (__any_sync(0xffffffffu, cm > mu + 8.f)) {
        const float nm = cm > mu + 8.f ? cm : mu;
        const float beta = nm == mu ? 1.f : exp2f(mu - nm);
        mu = nm;
        psum *= beta;
        alpha *= beta;
        tmem_wait_st();  // the P stored so far, before it is read back or replaced
        if (c0 > 0) {
#pragma unroll 1
          for (int cc = 0; cc < (c0 >> 1); cc += 16) {
            uint32_t pv[16];
            tmem_ld16(tS + lane_base + cc, pv);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j)
              pv[j] = pack_bf16x2(bf16_lo(pv[j]) * beta, bf16_hi(pv[j]) * beta);
            tmem_st16(tS + lane_base + cc, pv);
          }
        }
        ps = p_chunk(x, mu, w);
        tmem_st16(tS + lane_base + (c0 >> 1), w);
      }
      psum += ps;
    }
    st.m_used = mu;
  }
  if (t > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
    for (int c0 = 0; c0 < kD; c0 += 32) {
      uint32_t v[32];
      tmem_ld32(tO + lane_base + c0, v);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * alpha);
      tmem_st32(tO + lane_base + c0, v);
    }
  }
  tmem_wait_st();
  st.l = st.l * alpha + psum;
}

// One work item: a pair of query tiles of one (sequence, kv head).  All roles
// of a CTA derive the same values from the same inputs, so they skip the same
// items and agree on every barrier phase.
struct Item {
  bool valid;
  int b, g, nA, nB;
  long long q0, nq, qtA, qtB, first_pos, spanned;
  int off;
  int t0, c;  // shared-prefix prefix pass: first key tile and split index
};

__device__ __forceinline__ Item make_item(const PfParams& p, long long i, int tid) {
  Item it{};
  const long long per = (long long)p.batch * p.hkv;
  const long long px = i / per;  // pair rank: 0 = the latest (heaviest) pair
  const long long rem = i - px * per;
  it.b = (int)(rem / p.hkv);
  it.g = (int)(rem - (long long)it.b * p.hkv);
  it.q0 = p.cu_q[it.b];
  const long long q1 = p.cu_q[it.b + 1];
  it.nq = q1 - it.q0;
  if (it.nq <= 0) return it;
  const int TQ = p.TQ;
  const long long ntq = (it.nq + TQ - 1) / TQ;
  if (px >= (ntq + 1) / 2) return it;
  const long long len = p.lens[it.b];
  it.off = p.offs ? p.offs[it.b] : 0;
  if (it.nq > p.max_q_len || len < it.nq || it.off < 0 || it.off >= p.bs || q1 > p.total_q ||
      (long long)it.off + len > (long long)p.mb * p.bs) {
    // reported once, by the item of the sequence's first pair and head
    if (px == 0 && it.g == 0 && tid == 0) set_error(p.err, kErrCapacity);
    return it;
  }
  it.qtB = ntq - 1 - 2 * px;
  it.qtA = it.qtB - 1;
  it.first_pos = len - it.nq;
  auto tiles_for = [&](long long qt) -> int {
    if (qt < 0) return 0;
    const long long last = min(it.nq, (qt + 1) * TQ) - 1;
    return (int)((it.off + it.first_pos + last) / kKeys) + 1;
  };
  it.nA = tiles_for(it.qtA);
  it.nB = tiles_for(it.qtB);
  it.spanned = ((long long)it.off + len + p.bs - 1) / p.bs;
  it.valid = true;
  return it;
}

// Prefix pass of shared-prefix decode: item i is (query-tile pair px, key
// split c, kv head g).  Tile B = 2 px always exists, tile A = 2 px + 1 when
// the batch has it; both attend to the key tiles [t0, t0 + nB) of the
// prefix, read through table row 0 (every sequence's table starts with the
// same prefix blocks).  Per-row key masks come from each sequence's offset
// and length (softmax).
__device__ __forceinline__ Item make_item_prefix(const PfParams& p, long long i) {
  Item it{};
  const long long per = (long long)p.nsplit * p.hkv;
  const long long px = i / per;
  const long long rem = i - px * per;
  it.c = (int)(rem / p.hkv);
  it.g = (int)(rem - (long long)it.c * p.hkv);
  it.b = 0;
  it.q0 = 0;
  it.nq = p.batch;
  const long long ntq = (it.nq + p.TQ - 1) / p.TQ;
  if (px >= (ntq + 1) / 2) return it;
  it.t0 = it.c * p.per_split;
  const int nkt = min(p.key_tiles, it.t0 + p.per_split) - it.t0;
  if (nkt <= 0) return it;
  it.qtB = 2 * px;
  it.qtA = 2 * px + 1;
  it.nB = nkt;
  it.nA = it.qtA < ntq ? nkt : 0;
  it.spanned = p.prefix_blocks;
  it.valid = true;
  return it;
}

// CTA pairs: cluster item c gives the pair the query-tile pairs 2 c' and
// 2 c' + 1 of one (sequence, kv head) (c' = c / (batch x Hkv)); the even CTA
// holds the later pair, whose key tiles cover the other's.
__device__ __forceinline__ long long item_of(const PfParams& p, long long c, uint32_t rank) {
  const long long per = (long long)p.batch * p.hkv;
  const long long pc = c / per;
  return (2 * pc + rank) * per + (c - pc * per);
}

// Persistent: one CTA per SM walks the items c, c + grid, c + 2 grid, ...
// (pairs of every sequence and head in order of decreasing key count).  The
// K/V ring, the barrier phases and the TMEM allocation carry over from item
// to item, so the next item's loads and first products overlap the previous
// item's epilogue.
//
// CTA pairs (SHARE: clusters of two CTAs, one per SM, each computing its own
// items as above) read every K/V tile from L2 once for both CTAs:
//  * the two CTAs take neighbouring query-tile pairs of the same (sequence,
//    kv head) and stream the same key tiles (those of the even CTA's item;
//    the odd CTA's products skip the ones its item does not reach);
//  * each CTA loads by TMA one 64-column half of every tile (the even CTA
//    half 0, the odd one half 1) into its own ring, and its warp 10 then
//    copies that half into the same slot of the other CTA (a shared-memory
//    bulk copy between the CTAs), so each slot fills from both sides;
//  * a slot is refilled once the products of both CTAs have read it: every
//    release (a product commit, or an arrive for a tile not multiplied)
//    arrives on the "slot free" barriers of both CTAs.
// Each CTA waits for every release of its slots before it leaves (so no
// copy or arrive of the other CTA still targets it), and the two leave
// together (a cluster barrier).
template <bool PREFIX, bool SHARE>
__global__ void __launch_bounds__(pf_threads<SHARE>(), 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, const PfParams p) {
  static_assert(!(PREFIX && SHARE), "the prefix pass runs on single CTAs");
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // Prefix pass of shared-prefix decode: it reads nothing the grid before it
  // (the suffix pass) writes, and that grid's own inputs were complete when
  // it let this one launch, so its CTAs start as soon as the suffix pass
  // frees their SMs; each waits for the suffix pass only before it exits, so
  // the combine after this grid still sees both.
  if constexpr (!PREFIX) griddep_wait();
  griddep_launch_dependents();
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int TQ = p.TQ, G = p.G;
  const int blocks_per_tile = kKeys / p.bs;

  // ---- shared memory, barriers, TMEM --------------------------------------------------
  unsigned char* sQ = smem + kOffQ;  // [A | B]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + kOffTslot);
  // barriers: Q full, ring full[kSlots], ring empty[kSlots], then per tile
  // A / B: S ready, P written, O += P V done, O read by the epilogue, then
  // (CTA pairs) this CTA's own half of a slot loaded[kSlots]
  static_assert((3 * kSlots + 12 + 2 * kItemRing) * 8 <= kOffTslot - kOffBar,
                "barriers overlap the TMEM address slot");
  static_assert(kItemRing * 2 * sizeof(Item) <= 1024, "item ring overflows its carve");
  const uint32_t b_qfull = smem_addr(&bars[0]);
  const uint32_t b_full0 = smem_addr(&bars[1]);                // ring slot filled
  const uint32_t b_empty0 = smem_addr(&bars[1 + kSlots]);      // ring slot consumed
  const uint32_t b_sfull0 = smem_addr(&bars[1 + 2 * kSlots]);  // S of tile A / B ready
  const uint32_t b_pfull0 = smem_addr(&bars[3 + 2 * kSlots]);  // P of tile A / B written
  const uint32_t b_pvdone0 = smem_addr(&bars[5 + 2 * kSlots]); // O += P V of A / B done
  const uint32_t b_ofree0 = smem_addr(&bars[7 + 2 * kSlots]);  // O of A / B read by the epilogue
  const uint32_t b_drain = smem_addr(&bars[9 + 2 * kSlots]);
  const uint32_t b_qempty = smem_addr(&bars[10 + 2 * kSlots]);  // an item's S products read Q
  const uint32_t b_stall = smem_addr(&bars[11 + 2 * kSlots]);   // never arrived at (test hook)
  const uint32_t b_half0 = smem_addr(&bars[12 + 2 * kSlots]);   // own half of a slot loaded
  // the items' values, computed by the loads warp (which runs ahead) and read
  // by the MMA warp, whose thread must keep issuing products
  const uint32_t b_ifull0 = smem_addr(&bars[12 + 3 * kSlots]);
  const uint32_t b_iempty0 = smem_addr(&bars[12 + 3 * kSlots + kItemRing]);
  Item* s_items = reinterpret_cast<Item*>(smem + kOffItems);
  auto slot_full = [&](int i) { return b_full0 + 8u * i; };
  auto slot_empty = [&](int i) { return b_empty0 + 8u * i; };
  auto slot_half = [&](int i) { return b_half0 + 8u * i; };
  const uint32_t rank = SHARE ? cluster_rank() : 0u, peer = rank ^ 1u;
  auto slot_ptr = [&](int i) { return smem + kOffKV + i * kTileBytes; };

  if (tid == 0) {
    mbar_init(b_qfull, 1);
    mbar_init(b_qempty, 1);
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(slot_full(i), 1);
      mbar_init(slot_empty(i), SHARE ? 2 : 1);  // a pair: released by both CTAs
      mbar_init(slot_half(i), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(b_sfull0 + 8u * x, 1);
      mbar_init(b_pfull0 + 8u * x, 4);
      mbar_init(b_pvdone0 + 8u * x, 1);
      mbar_init(b_ofree0 + 8u * x, 4);
    }
    mbar_init(b_drain, 1);
    mbar_init(b_stall, 1);
    for (int r = 0; r < kItemRing; ++r) {
      mbar_init(b_ifull0 + 8u * r, 1);
      mbar_init(b_iempty0 + 8u * r, 1);
    }
    fence_mbar_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tslot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  // CTA pair: the other CTA's copies and arrivals target these barriers
  if constexpr (SHARE) cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  // TMEM columns: S_A [0,128), S_B [128,256), O_A [256,384), O_B [384,512)
  auto tS = [&](int x) { return tmem + 128u * x; };
  auto tO = [&](int x) { return tmem + 256u + 128u * x; };
  const long long n_items = p.n_items;
  const long long i_first = SHARE ? blockIdx.x >> 1 : blockIdx.x;
  const long long i_step = SHARE ? gridDim.x >> 1 : gridDim.x;
  // this CTA's item of (cluster) item c, and the item whose key tiles the
  // pair streams (the even CTA's)
  auto own_item = [&](long long c) {
    return PREFIX ? make_item_prefix(p, c) : make_item(p, SHARE ? item_of(p, c, rank) : c, tid);
  };
  auto lead_item = [&](long long c, const Item& own) {
    return !SHARE || rank == 0 ? own : make_item(p, item_of(p, c, 0), tid);
  };
  const WaitCtl w = make_wait_ctl(p.err, p.wait_ns, p.epoch);
  bool ok = true;

  if (warp == kWarpTma) {
    // ================= TMA producer: per item Q, then K(0) V(0) K(1) V(1) ... =================
    const int box_bytes = p.bs * 128;
    long long ld = 0;  // K / V loads issued so far (ring position)
    int jq = 0;        // items whose Q was loaded
    long long ni = 0;  // items published
    for (long long i = i_first; i < n_items && ok; i += i_step, ++ni) {
      const Item it = own_item(i);
      const Item lead = lead_item(i, it);
      {
        const int r = (int)(ni % kItemRing);
        const long long use = ni / kItemRing;
        if (use > 0 && !mbar_wait_sleep(b_iempty0 + 8u * r, (uint32_t)((use - 1) & 1), w)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          s_items[2 * r] = it;
          s_items[2 * r + 1] = lead;
          mbar_arrive(b_ifull0 + 8u * r);
        }
      }
      if (!lead.valid) continue;
      if (it.valid) {
        // Q of this item once the previous item's S products have read the old one
        if (jq > 0 && !mbar_wait_sleep(b_qempty, (jq - 1) & 1, w)) { ok = false; break; }
        if (lane == 0) {
          mbar_arrive_expect_tx(b_qfull, (it.nA > 0 ? 2 : 1) * kTileBytes);
          for (int x = (it.nA > 0 ? 0 : 1); x < 2; ++x) {
            const int z = (int)(it.q0 + (x == 0 ? it.qtA : it.qtB) * TQ);
            for (int h = 0; h < 2; ++h)
              tma_3d(smem_addr(sQ + x * kTileBytes + h * kHalf), &tq, h * 64, it.g * G, z,
                     b_qfull);
          }
        }
        ++jq;
      }
      for (int li = 0; li < 2 * lead.nB && ok; ++li, ++ld) {
        const int slot = (int)(ld % kSlots);
        const long long use = ld / kSlots;
        if (use > 0 && !mbar_wait_sleep(slot_empty(slot), (uint32_t)((use - 1) & 1), w)) {
          ok = false;
          break;
        }
        const int t = li >> 1, is_v = li & 1;
        // one CTA: both 64-column halves; a pair: this CTA's half, counted on
        // its own "half loaded" barrier (the other half comes from the peer)
        const uint32_t bar = SHARE ? slot_half(slot) : slot_full(slot);
        if (lane == 0) mbar_arrive_expect_tx(bar, SHARE ? kHalf : kTileBytes);
        __syncwarp();
        for (int k2 = lane; k2 < (SHARE ? 1 : 2) * blocks_per_tile; k2 += 32) {
          const int h = SHARE ? (int)rank : k2 / blocks_per_tile;
          const int k = SHARE ? k2 : k2 % blocks_per_tile;
          const long long lb = (long long)(PREFIX ? lead.t0 + t : t) * blocks_per_tile + k;
          long long coord = p.blk_coord_limit;                       // out of range: zeros
          if (lb < lead.spanned) {
            const int blk = p.bt[(long long)lead.b * p.mb + lb];
            if (blk >= 0 && blk < p.num_blocks) {
              coord = (long long)blk * p.L + p.layer;
            } else {
              set_error(p.err, kErrIndex);
            }
          }
          tma_4d(smem_addr(slot_ptr(slot) + h * kHalf + k * box_bytes), is_v ? &tv : &tk, h * 64,
                 lead.g, 0, (int)coord, bar);
        }
        __syncwarp();
      }
    }
    // Every load issued must land before the CTA may leave: when the other
    // warps gave up, nothing else waited for the last ones.  A slot holds at
    // most one load in flight (it is refilled only after its release), so the
    // last load of each slot and the last Q load are the ones to wait for.
    for (long long idx = ld - kSlots; idx < ld; ++idx) {
      if (idx < 0) continue;
      const int slot = (int)(idx % kSlots);
      const uint32_t ph = (uint32_t)((idx / kSlots) & 1);
      if constexpr (SHARE) {
        // this CTA's own copies, then every release of the slot by both CTAs
        // (after which the other CTA sends nothing more into it)
        mbar_wait_drain(slot_half(slot), ph, p.err);
        mbar_wait_sleep(slot_empty(slot), ph, w);
      } else {
        mbar_wait_drain(slot_full(slot), ph, p.err);
      }
    }
    if (jq > 0) mbar_wait_drain(b_qfull, (uint32_t)((jq - 1) & 1), p.err);
  } else if (SHARE && warp == kWarpFwd) {
    // ================= CTA pair: this CTA's half of each slot to the other CTA =================
    // once its copy landed; this CTA's "slot full" then waits only for the
    // other CTA's half
    if (lane == 0) {
      const uint32_t half_off = rank * kHalf;
      long long ld = 0;
      for (long long i = i_first; i < n_items && ok; i += i_step) {
        const Item lead = lead_item(i, own_item(i));
        if (!lead.valid) continue;
        for (int li = 0; li < 2 * lead.nB; ++li, ++ld) {
          const int slot = (int)(ld % kSlots);
          if (!mbar_wait_sleep(slot_half(slot), (uint32_t)((ld / kSlots) & 1), w)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(slot_full(slot), kHalf);
          const uint32_t src = smem_addr(slot_ptr(slot)) + half_off;
          bulk_s2s(peer_addr(src, peer), src, kHalf, peer_addr(slot_full(slot), peer));
        }
      }
    }
  } else if (warp == kWarpMma) {
    // ================= MMA issuer =================
    // per item: S_A(0) S_B(0) | PV_A(t) S_A(t+1) PV_B(t) S_B(t+1) | ..., so
    // each warpgroup's softmax overlaps the other tile's products
    if (lane == 0) {
      if (p.skip_fill == 2 || (p.skip_fill == 1 && blockIdx.x == 0)) {
        // test hook: a wait on a barrier nothing arrives at, which can only
        // give up at the bound; no product is issued, so the other warps'
        // waits give up in turn
        mbar_wait_sleep(b_stall, 0, w);
        ok = false;
      }
      const uint32_t q_addr = smem_addr(sQ);
      long long ld = 0;            // K / V loads consumed so far
      int jq = 0;                  // items started
      long long nt[2] = {0, 0};    // tiles of A / B across items (barrier phases)
      int ne[2] = {0, 0};          // epilogues of A / B across items
      auto slot_of = [&](long long idx) { return (int)(idx % kSlots); };
      // A slot's "full" barrier completes on this CTA's own arrival and on the
      // transaction bytes of copies (this CTA's TMA loads; in a pair, the
      // other CTA's bulk copy into this CTA): completions of asynchronous
      // copies, which a CTA-scope wait orders before the products that read
      // the slot, as for any TMA load.
      auto ready = [&](long long idx) {
        return mbar_wait_sleep(slot_full(slot_of(idx)), (uint32_t)((idx / kSlots) & 1), w);
      };
      // a slot is free once the products reading it completed (in both CTAs
      // of a pair)
      auto release = [&](long long idx) {
        if constexpr (SHARE) {
          umma_commit_both(slot_empty(slot_of(idx)));
        } else {
          umma_commit(slot_empty(slot_of(idx)));
        }
      };
      // One thread issues every product, and a K = 16 step takes the tensor
      // cores only about 100 cycles, so the issue loop is kept short: each
      // product builds its two descriptors once and steps them by constants
      // (the start address is the descriptor's low field, in 16-byte units;
      // shared addresses stay below 256 KB, so the addition never carries).
      auto issue_s = [&](int x, long long k_idx) {
        const uint64_t a0 = desc_sw128(q_addr + x * kTileBytes, 16, 1024);
        const uint64_t b0 = desc_sw128(smem_addr(slot_ptr(slot_of(k_idx))), 16, 1024);
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t step = (uint64_t)(((k >> 2) * kHalf + (k & 3) * 32) >> 4);
          umma(tS(x), a0 + step, b0 + step, kIdescKK, k > 0);
        }
        umma_commit(b_sfull0 + 8u * x);
      };
      auto issue_pv = [&](int x, long long v_idx, bool first) {
        const uint64_t b0 = desc_sw128(smem_addr(slot_ptr(slot_of(v_idx))), kHalf, 1024);
        const uint32_t p0 = tS(x), o0 = tO(x);
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          // A = P from TMEM (S columns of tile x), B = V MN-major
          umma_ts(o0, p0 + 8u * k, b0 + (uint64_t)((k * 2048) >> 4), kIdescKMN,
                  (!first || k > 0) ? 1u : 0u);
        }
        umma_commit(b_pvdone0 + 8u * x);
      };
      long long ni = 0;  // items read from the loads warp
      for (long long i = i_first; i < n_items && ok; i += i_step, ++ni) {
        const int r = (int)(ni % kItemRing);
        if (!mbar_wait_sleep(b_ifull0 + 8u * r, (uint32_t)((ni / kItemRing) & 1), w)) {
          ok = false;
          break;
        }
        const Item it = s_items[2 * r];
        const Item lead = s_items[2 * r + 1];
        mbar_arrive(b_iempty0 + 8u * r);
        if (!lead.valid) continue;
        const int nA = it.valid ? it.nA : 0, nB = it.valid ? it.nB : 0;
        const long long base = ld;  // load index of K(0) of this item
        ld = base + 2 * lead.nB;
        if (it.valid) {
          if (!mbar_wait_sleep(b_qfull, jq & 1, w) || !ready(base)) { ok = false; break; }
          ++jq;
          if (nA > 0) issue_s(0, base);
          issue_s(1, base);
          // Q may be replaced once the last S product of the item completes: the
          // next item's loads then overlap this item's last products and epilogue
          if (nB == 1) umma_commit(b_qempty);
          for (int t = 0; t < nB && ok; ++t) {
            const long long ki = base + 2 * t, vi = ki + 1;
            // K(t) is released after the S products that read it
            release(ki);
            if (!ready(vi)) { ok = false; break; }
            if (t < nA) {
              // O_A is overwritten by the first product: the previous epilogue
              // must have read it
              if (t == 0 && ne[0] > 0 && !mbar_wait_sleep(b_ofree0, (ne[0] - 1) & 1, w)) {
                ok = false;
                break;
              }
              if (!mbar_wait_sleep(b_pfull0, (uint32_t)(nt[0] & 1), w)) { ok = false; break; }
              ++nt[0];
              issue_pv(0, vi, t == 0);
              if (t + 1 < nA) {
                if (!ready(ki + 2)) { ok = false; break; }
                issue_s(0, ki + 2);
              }
            }
            if (t == 0 && ne[1] > 0 && !mbar_wait_sleep(b_ofree0 + 8u, (ne[1] - 1) & 1, w)) {
              ok = false;
              break;
            }
            if (!mbar_wait_sleep(b_pfull0 + 8u, (uint32_t)(nt[1] & 1), w)) { ok = false; break; }
            ++nt[1];
            issue_pv(1, vi, t == 0);
            release(vi);
            if (t + 1 < nB) {
              if (!(t + 1 < nA) && !ready(ki + 2)) { ok = false; break; }
              issue_s(1, ki + 2);
              if (t + 2 == nB) umma_commit(b_qempty);
            }
          }
          if (nA > 0) ++ne[0];
          ++ne[1];
        }
        // tiles only the other CTA's item reads: wait for them and release
        // them in both CTAs
        for (int li = 2 * nB; li < 2 * lead.nB && ok; ++li) {
          const long long idx = base + li;
          if (!ready(idx)) { ok = false; break; }
          mbar_arrive(slot_empty(slot_of(idx)));
          mbar_arrive_remote(peer_addr(slot_empty(slot_of(idx)), peer));
        }
      }
      umma_commit(b_drain);  // arrives once every MMA issued above has completed
    }
  } else {
    // ================= softmax: warpgroup x = 0 (tile A) or 1 (tile B), one row per thread ======
    const int x = warp >> 2;
    const int r = tid & 127;                 // MMA row = TMEM lane
    const int qtok = r / G, hh = r - qtok * G;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t b_sfull = b_sfull0 + 8u * x, b_pfull = b_pfull0 + 8u * x;
    const uint32_t b_pvdone = b_pvdone0 + 8u * x, b_ofree = b_ofree0 + 8u * x;
    long long nt = 0;  // tiles of this warpgroup across items (barrier phases)
    for (long long i = i_first; i < n_items && ok; i += i_step) {
      const Item it = own_item(i);
      if (!it.valid) continue;
      const int nX = x == 0 ? it.nA : it.nB;
      if (nX == 0) continue;
      const long long qt = x == 0 ? it.qtA : it.qtB;
      const long long qi = qt * TQ + qtok;   // query index within the sequence
      const bool row_ok = qi < it.nq;
      const long long pos = it.first_pos + qi;  // its logical position
      // tiles before the first diagonal tile are full for every row when the
      // tile has no padding rows (and t = 0 only without a first-block offset)
      const int t_mask_lo = (int)((it.off + it.first_pos + qt * TQ) / kKeys);
      const bool rows_full = (qt + 1) * TQ <= it.nq;
      // prefix pass: the row is the decode query of sequence qi, whose keys
      // in the prefix are the table positions [key_lo, key_hi) (its offset
      // up to the end of its tokens or of the prefix); a sequence whose
      // offset or length is out of range has none
      long long key_lo = 0, key_hi = 0;
      if (PREFIX && row_ok) {
        const long long ob = p.offs ? p.offs[qi] : 0;
        const long long lb = p.lens[qi];
        if (ob >= 0 && ob < p.bs && lb >= 0 && ob + lb <= (long long)p.mb * p.bs) {
          key_lo = ob;
          key_hi = min((long long)p.prefix_blocks * p.bs, ob + lb);
        }
      }
      RowState st{-INFINITY, 0.f};
      for (int t = 0; t < nX && ok; ++t, ++nt) {
        const bool waited = mbar_wait_sleep(b_sfull, (uint32_t)(nt & 1), w);
        if (!__all_sync(0xffffffffu, waited)) { ok = false; break; }
        tc_fence_after();
        int c_lo, c_hi;
        bool full_tile;
        if constexpr (PREFIX) {
          const long long tp0 = (long long)(it.t0 + t) * kKeys;
          c_lo = (int)max(0ll, key_lo - tp0);
          c_hi = (int)max(-1ll, min((long long)kKeys - 1, key_hi - 1 - tp0));
          // warp-uniform: the tile is full only if it is for every row of the warp
          full_tile = __all_sync(0xffffffffu, c_lo == 0 && c_hi == kKeys - 1);
        } else {
          const long long tp0 = (long long)t * kKeys;
          c_lo = (int)max(0ll, (long long)it.off - tp0);
          c_hi = row_ok ? (int)min((long long)kKeys - 1, pos + it.off - tp0) : -1;
          full_tile = (t > 0 || it.off == 0) && t < t_mask_lo && rows_full;
        }
        softmax_tile(tS(x), tO(x), lane_base, t, c_lo, c_hi, full_tile, p.qscale, st);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_pfull);
      }
      if (!ok) break;
      // epilogue: O row / l -> bf16 -> out, then hand O back to the MMA warp
      const bool waited = mbar_wait_sleep(b_pvdone, (uint32_t)((nt - 1) & 1), w);
      if (!__all_sync(0xffffffffu, waited)) { ok = false; break; }
      tc_fence_after();
      if constexpr (PREFIX) {
        // the row's state (m, l, unnormalised O) for the decode combine
        const long long row = ((long long)it.c * p.batch + qi) * p.hq + (long long)it.g * G + hh;
        if (row_ok) {
          p.pre_ml[2 * row] = st.m_used;
          p.pre_ml[2 * row + 1] = st.l;
        }
        float* arow = p.pre_acc + row * kD;
#pragma unroll 1
        for (int c0 = 0; c0 < kD; c0 += 32) {
          uint32_t v[32];
          tmem_ld32(tO(x) + lane_base + c0, v);
          tmem_wait_ld();
          if (row_ok) {
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              *reinterpret_cast<uint4*>(arow + c0 + j) = make_uint4(v[j], v[j + 1], v[j + 2],
                                                                    v[j + 3]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_ofree);
        continue;
      }
      const float inv = st.l > 0.f ? 1.f / st.l : 0.f;
      __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.out) +
                            ((it.q0 + qi) * p.hq + (long long)it.g * G + hh) * kD;
#pragma unroll 1
      for (int c0 = 0; c0 < kD; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tO(x) + lane_base + c0, v);
        tmem_wait_ld();
        if (row_ok) {
          if ((reinterpret_cast<uintptr_t>(p.out) & 31) == 0) {
            // 32-byte stores (full sectors) when the output allows them
#pragma unroll
            for (int j = 0; j < 32; j += 16) {
              uint32_t o[8];
#pragma unroll
              for (int k = 0; k < 8; ++k)
                o[k] = pack_bf16x2(__uint_as_float(v[j + 2 * k]) * inv,
                                   __uint_as_float(v[j + 2 * k + 1]) * inv);
              asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(orow + c0 + j),
                           "r"(o[0]), "r"(o[1]), "r"(o[2]), "r"(o[3]), "r"(o[4]), "r"(o[5]),
                           "r"(o[6]), "r"(o[7])
                           : "memory");
            }
          } else {
#pragma unroll
          for (int j = 0; j < 32; j += 8) {
            uint4 o;
            o.x = pack_bf16x2(__uint_as_float(v[j]) * inv, __uint_as_float(v[j + 1]) * inv);
            o.y = pack_bf16x2(__uint_as_float(v[j + 2]) * inv, __uint_as_float(v[j + 3]) * inv);
            o.z = pack_bf16x2(__uint_as_float(v[j + 4]) * inv, __uint_as_float(v[j + 5]) * inv);
            o.w = pack_bf16x2(__uint_as_float(v[j + 6]) * inv, __uint_as_float(v[j + 7]) * inv);
            *reinterpret_cast<uint4*>(orow + c0 + j) = o;
          }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_ofree);
    }
  }

  // ---- teardown: every MMA this CTA issued has completed before TMEM is freed ----
  tc_fence_before();
  __syncthreads();
  if (warp == 0) mbar_wait_drain(b_drain, 0, p.err);
  // CTA pair: neither CTA leaves while the other may still address it
  if constexpr (SHARE) cluster_sync_all();
  if (warp == 0) {
    __syncwarp();  // the dealloc below is warp-wide
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
  if constexpr (PREFIX) griddep_wait();
}

// ---- host side ------------------------------------------------------------------

}  // namespace

int prefill_supported(const PoolView& pv, int num_q_heads) {
  if (pv.elem_size != 2 || pv.head_dim != kD) return 1;
  if (pv.block_size < 8 || pv.block_size > kKeys || kKeys % pv.block_size) return 1;
  if (num_q_heads % pv.num_kv_heads) return 1;
  const int G = num_q_heads / pv.num_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16) return 1;
  return 0;
}

namespace {

// Tensor maps and the common parameters of a prefill-kernel launch: q as
// (d, q head, token) boxes of (64, G, TQ), the pool as (d, kv head, row,
// block*L + layer) boxes of one block per 64-column half.
cudaError_t prefill_setup(const PoolView& pv, int layer, const void* q, int num_q_heads,
                          float scale, const int32_t* bt, int mb, const int32_t* lens,
                          const int32_t* offs, int batch, long long total_q, int* err,
                          CUtensorMap* tq, CUtensorMap* tk, CUtensorMap* tv, PfParams* pp) {
  const int G = num_q_heads / pv.num_kv_heads;
  const int TQ = kRows / G;
  {
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)num_q_heads, (cuuint64_t)total_q};
    cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)num_q_heads * kD * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)TQ};
    if (!encode_tiled(tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q, dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  const long long nl = pv.num_blocks * pv.num_layers;
  {
    cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)pv.num_kv_heads, (cuuint64_t)pv.block_size,
                          (cuuint64_t)nl};
    cuuint64_t strides[3] = {(cuuint64_t)kD * 2, (cuuint64_t)pv.row_bytes,
                             (cuuint64_t)pv.row_bytes * pv.block_size};
    cuuint32_t box[4] = {64, 1, (cuuint32_t)pv.block_size, 1};
    if (!encode_tiled(tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, pv.k, dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tiled(tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, pv.v, dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  PfParams p{};
  p.bt = bt;
  p.lens = lens;
  p.offs = offs;
  p.err = err;
  p.total_q = total_q;
  p.blk_coord_limit = nl;
  p.num_blocks = pv.num_blocks;
  p.mb = mb;
  p.batch = batch;
  p.hq = num_q_heads;
  p.hkv = pv.num_kv_heads;
  p.G = G;
  p.TQ = TQ;
  p.bs = pv.block_size;
  p.L = pv.num_layers;
  p.layer = layer;
  p.qscale = scale * kLog2e;
  p.wait_ns = wait_limit_ns();
  p.epoch = next_launch_epoch();
  p.skip_fill = debug_skip_fill();
  *pp = p;
  return cudaSuccess;
}

template <bool PREFIX>
cudaError_t prefill_launch(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const PfParams& p, int sm_count, cudaStream_t s) {
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && configured[dev] == 0) {
    e = cudaFuncSetAttribute(prefill_kernel<PREFIX, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  const long long grid = p.n_items < sm_count ? p.n_items : sm_count;
  return launch_kernel(prefill_kernel<PREFIX, false>, dim3((unsigned)grid),
                       dim3(pf_threads<false>()), (size_t)kSmemBytes, s, true, tq, tk, tv, p);
}

// CTA pairs: clusters of two CTAs, as many as can be resident at once (at
// most one per two SMs), as a programmatic dependent of the work before.
cudaError_t prefill_launch_pairs(const CUtensorMap& tq, const CUtensorMap& tk,
                                 const CUtensorMap& tv, const PfParams& p, int sm_count,
                                 cudaStream_t s) {
  auto kern = prefill_kernel<false, true>;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(pf_threads<true>());
  cfg.dynamicSmemBytes = (size_t)kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  static int max_pairs[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (max_pairs[dev] == 0) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    // resident clusters: a persistent grid larger than this would queue
    cfg.gridDim = dim3(2 * (unsigned)(sm_count / 2 > 0 ? sm_count / 2 : 1));
    cfg.numAttrs = 1;  // the cluster shape alone
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess) return e;
    max_pairs[dev] = n > 0 ? n : 1;
  }
  long long np = sm_count / 2 < max_pairs[dev] ? sm_count / 2 : max_pairs[dev];
  if (np < 1) np = 1;
  if (p.n_items < np) np = p.n_items;
  cfg.gridDim = dim3((unsigned)(2 * np));
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, p);
}

}  // namespace

cudaError_t launch_prefill(const PoolView& pv, int layer, const void* q, int num_q_heads,
                           float scale, const int32_t* bt, int mb, const int32_t* lens,
                           const int32_t* offs, const int64_t* cu_q, int batch, long long total_q,
                           int max_q_len, void* out, int* err, int sm_count, cudaStream_t s) {
  if (batch == 0 || total_q == 0 || max_q_len == 0) return cudaSuccess;
  CUtensorMap tq, tk, tv;
  PfParams p;
  cudaError_t e = prefill_setup(pv, layer, q, num_q_heads, scale, bt, mb, lens, offs, batch,
                                total_q, err, &tq, &tk, &tv, &p);
  if (e != cudaSuccess) return e;
  p.cu_q = reinterpret_cast<const long long*>(cu_q);
  p.out = out;
  p.max_q_len = max_q_len;
  const long long ntq = (max_q_len + p.TQ - 1) / p.TQ;
  // CTA pairs: pairs of query-tile pairs per (sequence, kv head)
  p.n_items = ((ntq + 1) / 2 + 1) / 2 * (long long)batch * pv.num_kv_heads;
  return prefill_launch_pairs(tq, tk, tv, p, sm_count, s);
}

void prefix_plan(const PoolView& pv, int num_q_heads, int batch, int prefix_blocks, int sm_count,
                 int* nsplit, int* per_split) {
  const int G = num_q_heads / pv.num_kv_heads;
  const long long TQ = kRows / G;
  const long long ntq = (batch + TQ - 1) / TQ;
  const long long base = (ntq + 1) / 2 * pv.num_kv_heads;  // items of one key split
  const long long kt = ((long long)prefix_blocks * pv.block_size + kKeys - 1) / kKeys;
  long long want = base > 0 ? (sm_count + base - 1) / base : 1;  // splits that fill the GPU
  if (want < 1) want = 1;
  if (want > kt) want = kt;
  const long long ps = (kt + want - 1) / want;
  *per_split = (int)ps;
  *nsplit = (int)((kt + ps - 1) / ps);
}

cudaError_t launch_prefix_pass(const PoolView& pv, int layer, const void* q, int num_q_heads,
                               float scale, const int32_t* bt, int mb, const int32_t* lens,
                               const int32_t* offs, int batch, int prefix_blocks, float* pre_ml,
                               float* pre_acc, int* err, int sm_count, cudaStream_t s) {
  if (batch == 0 || prefix_blocks == 0) return cudaSuccess;
  CUtensorMap tq, tk, tv;
  PfParams p;
  cudaError_t e = prefill_setup(pv, layer, q, num_q_heads, scale, bt, mb, lens, offs, batch,
                                batch, err, &tq, &tk, &tv, &p);
  if (e != cudaSuccess) return e;
  int nsplit = 1, per_split = 1;
  prefix_plan(pv, num_q_heads, batch, prefix_blocks, sm_count, &nsplit, &per_split);
  p.prefix_blocks = prefix_blocks;
  p.key_tiles = (int)(((long long)prefix_blocks * pv.block_size + kKeys - 1) / kKeys);
  p.nsplit = nsplit;
  p.per_split = per_split;
  p.pre_ml = pre_ml;
  p.pre_acc = pre_acc;
  const long long ntq = (batch + p.TQ - 1) / p.TQ;
  p.n_items = (ntq + 1) / 2 * (long long)nsplit * pv.num_kv_heads;
  return prefill_launch<true>(tq, tk, tv, p, sm_count, s);
}

}  // namespace pkv
