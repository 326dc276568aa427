/*
 * pkv.h - C ABI of the GB300 paged KV cache library (libpkv.so).
 *
 * The library implements the data-parallel hot path of a paged KV cache:
 *   - the logical -> physical index step that turns (sequence, position)
 *     pairs into slot numbers      (pkv_build_slot_mapping),
 *   - the slot_mapping scatter     (pkv_write_slots),
 *   - the block_table gather       (pkv_gather),
 *   - fused paged decode attention that reads K/V through the block table
 *     with a split-K partial pass and a combine pass (pkv_decode_attention).
 *
 * Sources restated (cited by page title and section):
 *   [step14_2]  mini-vLLM tutorial "step14_2 - index_select gather"
 *   [vllm-notes] "vLLM PagedAttention source notes"
 *   [ch12]      mini-runtime "ch.12 Paged KV Cache"
 *
 * Conventions shared by every call
 *   Pool layout.  A pool descriptor names two caller-owned device tensors,
 *     k_cache and v_cache, each row-major [num_blocks, num_layers, block_size,
 *     num_kv_heads, head_dim] ([vllm-notes] §2.2, PagedKVCache paragraph: K
 *     and V held separately).  A token row (all kv heads of one token) of
 *     block b, layer l, row j starts at element ((b*L + l)*bs + j)*Hkv*D.
 *   Slots.  slot = block * block_size + row ([vllm-notes] §2.2); a slot
 *     addresses a row within one layer, the layer is a separate argument.
 *   Block tables.  int32 [batch, max_blocks_per_seq], row-major; entry k of
 *     row b is the physical block of logical block k of sequence b ([ch12]
 *     §2.2 BlockTable._block_ids).  offsets[b] (0 <= offsets[b] < block_size,
 *     NULL means all zero) is the first-block offset ([ch12] §2.2): logical
 *     token i of sequence b sits at table position p = offsets[b] + i, in
 *     block table[b][p / bs], row p % bs.  Capacity of a row of the table is
 *     max_blocks_per_seq * block_size - offsets[b] ([ch12] §2.2); entries past
 *     the blocks a sequence spans are never read.
 *   Memory.  Every pointer argument except `pool` itself is a DEVICE pointer
 *     owned by the caller; the descriptor struct is read on the host during
 *     the call only.  The library never allocates, frees or keeps device
 *     memory; scratch for the decode pass is the caller's workspace.
 *     k_cache, v_cache, k_new, v_new, k_out, v_out, q, out and workspace
 *     must be 16-byte aligned; index arrays must be naturally aligned.
 *   Streams.  Work is enqueued on `stream` (0 = the legacy default stream)
 *     and is asynchronous; nothing synchronises unless validate mode is on.
 *     The current CUDA device must be the device that owns the pointers.
 *   Errors.  Argument checks on host-visible values run before anything is
 *     enqueued and return a status without side effects.  Values that live
 *     in device memory (slots, block ids, offsets, lengths) are checked by
 *     the kernels themselves: an out-of-range index is never dereferenced;
 *     the access is skipped and a sticky device error word is set.  With
 *     validate mode on (pkv_set_validate), each call also runs a validation
 *     pass over its index inputs before the main kernel, synchronises the
 *     stream and returns PKV_ERR_INDEX / PKV_ERR_CAPACITY instead of running
 *     the main kernel; without it, pkv_device_error() reports the word.
 *     A failed CUDA launch returns PKV_ERR_CUDA.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = 1,  /* null pointer, bad size, bad layer, misaligned pointer */
  PKV_ERR_CAPACITY = 2,     /* a sequence does not fit its table row, or bad offset */
  PKV_ERR_UNSUPPORTED = 3,  /* shape or dtype outside the compiled kernels */
  PKV_ERR_WORKSPACE = 4,    /* workspace null or smaller than pkv_decode_workspace_size */
  PKV_ERR_INDEX = 5,        /* slot or block id outside the pool, bad packed layout */
  PKV_ERR_CUDA = 6,         /* a CUDA runtime call failed */
  PKV_ERR_TIMEOUT = 7,      /* a bounded device-side wait gave up */
  PKV_ERR_NO_BLOCKS = 8     /* allocator: too few free blocks; nothing was changed */
} pkv_status;

/* PKV_I8 is the quantised pool ([ch12] §6 Evolution names int8 KV as the
 * next step of paged caches; the scheme below is this library's reading).
 * Its token row (all kv heads of one token) is a byte row of
 *     R = num_kv_heads * head_dim + pad16(4 * num_kv_heads)
 * bytes: the num_kv_heads * head_dim codes (head-major, each stored offset
 * binary as the byte code + 128, codes in [-127, 127]), then one fp32 scale
 * per kv head (little-endian), then padding to a multiple of 16 bytes.  The
 * stored value of element d of head g is code[g][d] * scale[g]. */
typedef enum { PKV_F32 = 0, PKV_BF16 = 1, PKV_I8 = 2 } pkv_dtype;

/* Pool descriptor: two device tensors [num_blocks, num_layers, block_size,
 * num_kv_heads, head_dim] of `dtype` (PKV_I8: bytes [num_blocks, num_layers,
 * block_size, R], R as above).  block_size must be a power of two in
 * [1, 1024]; num_kv_heads * head_dim * element size must be a multiple of 16
 * bytes.  ([vllm-notes] §2.2 layout; [ch12] §4.2 uses block_size 16.) */
typedef struct {
  void* k_cache;
  void* v_cache;
  int64_t num_blocks;
  int32_t num_layers;
  int32_t block_size;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t dtype; /* pkv_dtype */
} pkv_pool;

/* Logical -> physical index ([vllm-notes] §2.2 slot_mapping definition;
 * [step14_2] "Solution": position // block_size and position % block_size;
 * [ch12] §2.2 first-block offset).
 *
 * For t < num_tokens: if token_seq[t] < 0 the entry is padding and
 * slot_mapping[t] = -1; otherwise with b = token_seq[t] and
 * p = offsets[b] + token_pos[t]:
 *     slot_mapping[t] = block_tables[b][p / bs] * bs + p % bs.
 * token_seq, token_pos: int32 [num_tokens]; slot_mapping: int64 [num_tokens]
 * (written).  offsets may be NULL.  A token whose position lies outside its
 * table row (p >= max_blocks_per_seq * bs, b >= batch, negative position) or
 * whose block id is outside [0, num_blocks) gets slot -1 and sets the device
 * error word (PKV_ERR_INDEX in validate mode). */
PKV_API pkv_status pkv_build_slot_mapping(const pkv_pool* pool, const int32_t* block_tables,
                                  int32_t max_blocks_per_seq, const int32_t* offsets,
                                  int32_t batch, const int32_t* token_seq,
                                  const int32_t* token_pos, int64_t num_tokens,
                                  int64_t* slot_mapping, cudaStream_t stream);

/* Scatter ([step14_2] "Relation to step14_1": kv_pool[blocks, rows] = K;
 * [vllm-notes] §2.2: rows addressed as [block_id, layer, offset], -1 = padding).
 *
 * For t < num_tokens with s = slot_mapping[t] >= 0:
 *     k_cache[s / bs][layer][s % bs] = k_new[t],  v_cache[...] = v_new[t].
 * k_new, v_new: [num_tokens, Hkv, D] in the pool dtype, contiguous.
 * PKV_I8 pools take bf16 k_new / v_new and quantise each (token, kv head)
 * row of D values x on the way in: scale = absmax(x) / 127 and
 * code = round_half_even(x / scale) clamped to [-127, 127], both divisions
 * IEEE fp32 round-to-nearest (subnormals kept); a row of zeros stores scale
 * 0 and codes 0.  The padding bytes of the row are not written.  For int8
 * pools head_dim must be 32, 64, 128 or 256 (else PKV_ERR_UNSUPPORTED).  Entries
 * equal to -1 are skipped and their rows untouched.  Other negative entries
 * and entries >= num_blocks * bs are skipped and set the device error word
 * (PKV_ERR_INDEX in validate mode).  Non-negative slots must be distinct; a
 * repeated slot leaves that row holding one of the written rows. */
PKV_API pkv_status pkv_write_slots(const pkv_pool* pool, int32_t layer, const void* k_new,
                           const void* v_new, const int64_t* slot_mapping,
                           int64_t num_tokens, cudaStream_t stream);

/* Slot mapping and scatter in one call: the new rows of a decode step (or a
 * prompt) go straight from (sequence, position) pairs into their slots.  The
 * result is that of pkv_build_slot_mapping followed by pkv_write_slots with
 * its output, in one kernel: for each token t, the slot is computed as in
 * pkv_build_slot_mapping (padding and out-of-range tokens get -1 and are not
 * written; out-of-range ones set the device error word, PKV_ERR_INDEX /
 * PKV_ERR_CAPACITY in validate mode) and row t of k_new / v_new is written
 * there as in pkv_write_slots (quantised for PKV_I8 pools).  slot_mapping
 * (int64 [num_tokens], device) receives the slots when not NULL.  Arguments
 * and their rules are those of the two calls. */
PKV_API pkv_status pkv_append_tokens(const pkv_pool* pool, int32_t layer,
                                     const int32_t* block_tables, int32_t max_blocks_per_seq,
                                     const int32_t* offsets, int32_t batch,
                                     const int32_t* token_seq, const int32_t* token_pos,
                                     int64_t num_tokens, const void* k_new, const void* v_new,
                                     int64_t* slot_mapping, cudaStream_t stream);

/* Gather ([step14_2] "Problem" and "Solution"; [vllm-notes] §2.3
 * gather_kv_for_attention; [ch12] §2.2 offset, §2.5 read_layer).
 *
 * For every sequence b and i < seq_lens[b], with p = offsets[b] + i:
 *     k_out[cu_seqlens[b] + i] = k_cache[block_tables[b][p / bs]][layer][p % bs]
 * and the same for V.  k_out, v_out: [total_tokens, Hkv, D] contiguous, pool
 * dtype (PKV_I8: the byte rows as stored, [total_tokens, R]).  cu_seqlens: int64 [batch + 1], the packed output layout, with
 * cu_seqlens[0] = 0, cu_seqlens[b+1] - cu_seqlens[b] = seq_lens[b] and
 * cu_seqlens[batch] = total_tokens (validate mode checks all three).
 * total_tokens is the number of output rows the caller allocated.  A row
 * whose block id is outside the pool, or which lies past its table row's
 * capacity, is left unwritten and sets the device error word. */
PKV_API pkv_status pkv_gather(const pkv_pool* pool, int32_t layer, const int32_t* block_tables,
                      int32_t max_blocks_per_seq, const int32_t* seq_lens,
                      const int32_t* offsets, int32_t batch, const int64_t* cu_seqlens,
                      int64_t total_tokens, void* k_out, void* v_out, cudaStream_t stream);

/* Bytes of workspace pkv_decode_attention needs for this shape on the
 * current device (it depends on the device's SM count).  0 on a bad shape. */
PKV_API size_t pkv_decode_workspace_size(int32_t batch, int32_t num_q_heads, int32_t head_dim);

/* Paged decode attention, one query token per sequence ([step14_2] comparison
 * with vLLM: attention reads the pool through the block table and K/V are
 * never copied to contiguous memory; [vllm-notes] §2.3 the same result as
 * gather + standard attention; [ch12] §3.1 PagedAttention).
 *
 * For each sequence b and query head h, with kv head g = h / (Hq / Hkv):
 *     s_i  = scale * dot(q[b][h], K_i[g])  over the seq_lens[b] tokens read
 *            through the table as in pkv_gather,
 *     out[b][h] = sum_i softmax(s)_i * V_i[g].
 * q, out: [batch, num_q_heads, head_dim] contiguous in the pool dtype.
 * seq_lens[b] == 0 gives an all-zero row.  Accumulation is fp32.
 * For PKV_I8 pools q and out are bf16 and K_i, V_i are the dequantised
 * rows (code * scale).  Both products run on fp16 tensor cores over the
 * exact codes: q is scaled by a power of two into fp16, and the V scales
 * are folded into the softmax weights (normalised by a running power of
 * two), which are rounded to fp16 for the P.V product.
 * The work is split along the sequence across the GPU; partial softmax
 * states go to `workspace` (>= pkv_decode_workspace_size bytes, contents
 * need no initialisation and are overwritten) and a second kernel combines
 * them.  Both kernels are launched as programmatic dependents of the work
 * before them on the stream and wait for it before reading any input, so the
 * call may be captured in a CUDA graph and replayed.  Supported: head_dim 64 or 128; num_kv_heads 1, 2, 4 or 8;
 * num_q_heads / num_kv_heads 1, 2, 4 or 8; any pool dtype; any block_size the
 * pool allows.  Others return PKV_ERR_UNSUPPORTED.  A sequence whose offset
 * is out of range or whose length exceeds its table row's capacity is
 * treated as empty and sets the device error word (PKV_ERR_CAPACITY in
 * validate mode); a block id outside the pool is skipped (PKV_ERR_INDEX). */
PKV_API pkv_status pkv_decode_attention(const pkv_pool* pool, int32_t layer, const void* q,
                                int32_t num_q_heads, float scale,
                                const int32_t* block_tables, int32_t max_blocks_per_seq,
                                const int32_t* seq_lens, const int32_t* offsets,
                                int32_t batch, void* out, void* workspace,
                                size_t workspace_bytes, cudaStream_t stream);

/* One decode step in one pass over the pool: for every sequence b with
 * seq_lens[b] > 0, the new token at logical position p = seq_lens[b] - 1
 * (already counted in seq_lens) has its K and V rows k_new[b], v_new[b]
 * stored at its slot table[b][(off + p) / bs] * bs + (off + p) % bs of
 * `layer` ([vllm-notes] §2.2 slot mapping and scatter; [step14_2] the
 * relation between writing the new K/V and reading them back), and decode
 * attention then runs over positions 0..p exactly as pkv_decode_attention.
 * The result equals pkv_append_tokens with token b at position
 * seq_lens[b] - 1, followed by pkv_decode_attention: same pool bytes, same
 * output.  The CTA of the attention kernel whose share of the blocks holds a
 * sequence's last block stores that sequence's new row before it starts
 * reading, so the step is one launch (plus the combine) instead of a
 * scatter launch followed by attention.
 * k_new, v_new: [batch, num_kv_heads, head_dim] contiguous in q's dtype
 * (bf16 for PKV_I8 pools, which quantise the new rows exactly as
 * pkv_write_slots does), device, 16-byte aligned (PKV_ERR_INVALID_ARG
 * otherwise).  Sequences with seq_lens[b] == 0 store nothing.  The new
 * token's block must not appear in another sequence's table in the same
 * call (copy-on-write guarantees it).  All other arguments, checks and errors
 * are those of pkv_decode_attention. */
PKV_API pkv_status pkv_decode_step(const pkv_pool* pool, int32_t layer, const void* q,
                                   int32_t num_q_heads, float scale,
                                   const int32_t* block_tables, int32_t max_blocks_per_seq,
                                   const int32_t* seq_lens, const int32_t* offsets,
                                   int32_t batch, const void* k_new, const void* v_new,
                                   void* out, void* workspace, size_t workspace_bytes,
                                   cudaStream_t stream);

/* Paged decode attention over a batch whose sequences share a prefix of
 * whole blocks (mini-runtime "ch.12 Paged KV Cache" §2.2: a sequence that
 * hits a cached prefix starts at an offset inside its first block; §2.4:
 * the prefix blocks are shared through their ref_count, not copied;
 * "vLLM PagedAttention source notes" §3: shared prefixes are why paging
 * wastes so little).  The result is that of pkv_decode_attention with the
 * same arguments; only the way the pool is read differs: the shared prefix is
 * read once for the whole batch instead of once per sequence.
 *
 * Contract: the first num_prefix_blocks entries of row 0 of block_tables
 * name the shared prefix blocks (all of them, even where sequence 0 ends
 * earlier), and every sequence's table agrees with row 0 on each of those
 * entries it spans (a sequence may end inside the prefix; its offset is its
 * first-block offset as usual).  Validate mode checks both (PKV_ERR_INDEX);
 * without it, a disagreeing table gives wrong results for that sequence and
 * an invalid id in row 0 reads zeros and sets the device error word (never
 * an out-of-range access).  0 <= num_prefix_blocks <=
 * max_blocks_per_seq, else PKV_ERR_INVALID_ARG.
 *
 * How it runs: a suffix pass (the decode partial kernel over the table
 * entries after the prefix), a prefix pass on the tcgen05 tensor cores (the
 * queries of all sequences, 128 / G sequences x G heads per MMA tile,
 * against the prefix's key tiles, split over the GPU; per-row masks from each
 * sequence's offset and length), and a combine of both by the log-sum-exp
 * rule.  That path needs bf16 pools with head_dim 128 and block_size 8..128
 * dividing 128, and batch <= 2048; for other shapes, or num_prefix_blocks ==
 * 0, the call runs pkv_decode_attention's path instead (same result).
 * workspace: >= pkv_decode_shared_prefix_workspace_size bytes (contents need
 * no initialisation).  All other arguments, checks and errors are those of
 * pkv_decode_attention. */
PKV_API size_t pkv_decode_shared_prefix_workspace_size(const pkv_pool* pool, int32_t batch,
                                                       int32_t num_q_heads,
                                                       int32_t num_prefix_blocks);
PKV_API pkv_status pkv_decode_attention_shared_prefix(const pkv_pool* pool, int32_t layer,
                                                      const void* q, int32_t num_q_heads,
                                                      float scale, const int32_t* block_tables,
                                                      int32_t max_blocks_per_seq,
                                                      const int32_t* seq_lens,
                                                      const int32_t* offsets, int32_t batch,
                                                      int32_t num_prefix_blocks, void* out,
                                                      void* workspace, size_t workspace_bytes,
                                                      cudaStream_t stream);

/* Paged prefill attention (the prefill batch of
 * "vLLM PagedAttention source notes" §2.4: the prompt tokens' K/V are written
 * into their blocks, then attention runs over them), on tcgen05 tensor cores.
 *
 * For each sequence b, the queries are its LAST n_b = cu_q[b+1] - cu_q[b]
 * tokens (their K/V must already be in the pool, e.g. by pkv_write_slots):
 * query i sits at logical position P = seq_lens[b] - n_b + i and attends
 * causally to the keys 0..P of the sequence, read through the block table
 * (first-block offset honoured):
 *     out[cu_q[b] + i][h] = sum_{j <= P} softmax_j(scale * q . K_j[g]) V_j[g],
 *     g = h / (num_q_heads / num_kv_heads).
 * q, out: [total_q, num_q_heads, head_dim] bf16 (device); cu_q: int64
 * [batch + 1] device, cu_q[0] = 0, nondecreasing, cu_q[batch] <= total_q;
 * max_q_len (host) bounds every n_b (the grid is sized from it; a sequence
 * with a larger n_b is skipped and sets the device error word).
 * A sequence with n_b > seq_lens[b] or a bad offset / capacity is skipped and
 * sets the error word (PKV_ERR_CAPACITY in validate mode).  Supported: bf16
 * pools with head_dim 128, block_size 8..128 dividing 128, num_q_heads /
 * num_kv_heads in {1, 2, 4, 8, 16}; others PKV_ERR_UNSUPPORTED.  No
 * workspace.  fp32 accumulation; P is rounded to bf16 for the P.V product.
 * The kernel runs as clusters of two CTAs (one per SM) whose CTAs share each
 * K/V tile; the grid holds as many clusters as can be resident at once. */
PKV_API pkv_status pkv_prefill_attention(const pkv_pool* pool, int32_t layer, const void* q,
                                         int32_t num_q_heads, float scale,
                                         const int32_t* block_tables, int32_t max_blocks_per_seq,
                                         const int32_t* seq_lens, const int32_t* offsets,
                                         const int64_t* cu_q, int32_t batch, int64_t total_q,
                                         int32_t max_q_len, void* out, cudaStream_t stream);

/* Allocation-free paged decode attention.  The paper has no counterpart:
 * this is a library convenience.  Same computation, arguments, results and
 * error behaviour as pkv_decode_attention, except that the caller passes no
 * workspace: the split-K scratch lives in a fixed device array defined inside
 * libpkv (PKV_DECODE_STATIC_SCRATCH_BYTES per GPU, held by every GPU that
 * loads the library until the process exits).
 *
 * It is meant for callers that cannot allocate device memory where they run
 * decode attention: serving processes whose memory manager reserves the
 * GPU's memory up front and hands out nothing on the hot path, plugin
 * runtimes whose execute step must not allocate, and plain C programs that
 * link only this library and have no device allocator for scratch.  The call
 * itself allocates nothing.
 *
 * Limits and rules:
 *   - A shape whose scratch (pkv_decode_workspace_size for the same batch,
 *     num_q_heads and head_dim) exceeds PKV_DECODE_STATIC_SCRATCH_BYTES is
 *     refused with PKV_ERR_WORKSPACE before anything is enqueued.
 *   - The first call on a device looks up the array's device address for that
 *     device; make that first call before any stream capture starts.
 *   - All calls on a device share the one array: calls whose kernels overlap
 *     on the GPU (different streams, or concurrent host threads) race and
 *     give wrong results.  Calls on one stream are ordered and safe.  The
 *     array keeps the previous call's contents; nothing in it needs to start
 *     at zero (every scratch word is written before it is read). */
#define PKV_DECODE_STATIC_SCRATCH_BYTES ((size_t)16 << 20)

PKV_API pkv_status pkv_decode_attention_static(const pkv_pool* pool, int32_t layer,
                                               const void* q, int32_t num_q_heads, float scale,
                                               const int32_t* block_tables,
                                               int32_t max_blocks_per_seq,
                                               const int32_t* seq_lens, const int32_t* offsets,
                                               int32_t batch, void* out, cudaStream_t stream);

/* Whole-block moves.  `layer` is one layer, or -1 for every layer of the
 * block (one contiguous run of num_layers * block_size rows).  Block ids
 * outside [0, num_blocks) are skipped and set the device error word
 * (PKV_ERR_INDEX in validate mode).
 *
 * pkv_copy_blocks: for i < num_pairs, block dst_blocks[i] receives the K and
 * V contents of block src_blocks[i] (device int32 arrays).  This is the copy
 * of copy-on-write (mini-runtime "ch.12 Paged KV Cache" §3.1; the allocator's
 * pkv_seq_append reports the pairs).  Destinations must be distinct and must
 * not appear among the sources. */
PKV_API pkv_status pkv_copy_blocks(const pkv_pool* pool, int32_t layer, const int32_t* src_blocks,
                                   const int32_t* dst_blocks, int32_t num_pairs,
                                   cudaStream_t stream);

/* pkv_swap_out: the K and V data of blocks[0..n) (device int32 array), in
 * that order, into host_k / host_v laid out [n, layers, block_size,
 * num_kv_heads, head_dim] (layers = 1 for a single layer; PKV_I8 pools:
 * [n, layers, block_size, R] bytes, codes and scales together).  pkv_swap_in: the
 * reverse, host buffers into the listed blocks.  Preemption by swapping
 * ("vLLM PagedAttention source notes" §2.4).  host_k and host_v must be
 * page-locked host memory the device can address (cudaHostAlloc or
 * cudaHostRegister; checked) of at least host_bytes bytes each, and
 * host_bytes must cover n blocks (checked); the kernel reads and writes them
 * in place, which on GB300 goes over NVLink-C2C. */
PKV_API pkv_status pkv_swap_out(const pkv_pool* pool, int32_t layer, const int32_t* blocks,
                                int32_t n, void* host_k, void* host_v, size_t host_bytes,
                                cudaStream_t stream);
PKV_API pkv_status pkv_swap_in(const pkv_pool* pool, int32_t layer, const int32_t* blocks,
                               int32_t n, const void* host_k, const void* host_v,
                               size_t host_bytes, cudaStream_t stream);

/* Number of CTAs the decode partial pass uses on the current device; 0 (the
 * default) means one per SM.  A positive value (at most 65536) forces that
 * grid size, which changes how sequences are split (1 = no split).
 * Process-wide. */
PKV_API pkv_status pkv_set_decode_ctas(int32_t num_ctas);

/* Profiling hook for the decode partial pass.  When both events are
 * non-null, each later pkv_decode_attention call records `start` on its
 * stream right before its first partial-pass kernel and `stop` right after
 * its last one (before the combine kernel), so the caller can time that
 * kernel alone with cudaEventElapsedTime.  Events are the caller's (created
 * with timing enabled); pass NULLs to stop recording.  Process-wide. */
PKV_API pkv_status pkv_set_decode_events(cudaEvent_t start, cudaEvent_t stop);

/* Bound on every device-side wait of the kernels (mbarrier waits between the
 * copy, tensor-core and softmax warps of one CTA), in nanoseconds of the GPU's
 * global timer; 0 restores the default (4 s).  Accepted range 1 us .. 60 s,
 * else PKV_ERR_INVALID_ARG.  A healthy wait lasts microseconds; the bound only
 * ends waits that can never complete.  The first wait of a launch to reach it
 * sets the timeout bit of the device error word (PKV_ERR_TIMEOUT in validate
 * mode or from pkv_device_error); every other pending wait of that launch
 * then gives up within a few polls, so the whole launch ends about one bound
 * after it stalled.  Copies a CTA has issued are always waited for (with the
 * default bound) before it exits.  The timeout bit stays set until cleared
 * (pkv_device_error with clear != 0, or a validate-mode call that reports
 * it).  Each launch carries its own number, so a give-up never cuts short a
 * later launch; the one exception is a launch replayed from a CUDA graph,
 * which keeps the number it was captured with: after such a replay gave up,
 * clear the error word before the next replay.  Process-wide; read at each
 * launch. */
PKV_API pkv_status pkv_set_wait_limit_ns(uint64_t ns);
PKV_API uint64_t pkv_get_wait_limit_ns(void);

/* Test hook for the give-up path, process-wide, default 0 (off).  With
 * mode 1 the first CTA, with mode 2 every CTA, of each decode partial pass
 * leaves its first pipeline stage unfilled, and of each prefill launch its
 * first K tile unloaded: nothing is copied into them, so the waits on them
 * can only give up at the wait bound.  Results of such launches are not
 * valid; the call reports PKV_ERR_TIMEOUT in validate mode.  Other modes:
 * PKV_ERR_INVALID_ARG.  Never needed outside tests. */
PKV_API pkv_status pkv_set_debug_skip_fill(int32_t mode);

/* Validate mode (process-wide, default off): see "Errors" above. */
PKV_API pkv_status pkv_set_validate(int32_t on);
PKV_API int32_t pkv_get_validate(void);

/* Synchronises the current device, stores the sticky device error word's
 * status (PKV_OK, PKV_ERR_INDEX, PKV_ERR_CAPACITY or PKV_ERR_TIMEOUT) in
 * *status and, if clear != 0, resets it.  Returns PKV_ERR_CUDA if the
 * device cannot be read. */
PKV_API pkv_status pkv_device_error(pkv_status* status, int32_t clear);

/* ------------------------------------------------------------------------
 * Host block allocator (block manager).  Plain host memory, no CUDA calls;
 * one allocator per pool; not thread-safe (the caller serialises calls).
 *
 * Restates mini-runtime "ch.12 Paged KV Cache" §2.2 (BlockTable: block ids in
 * logical order, first-block offset, capacity = blocks * block_size - offset),
 * §2.3 (FIFO deque of free ids: allocate takes ceil(tokens / block_size) ids
 * from the front, or fails and changes nothing), §2.4 (ref_count: inc_ref
 * when a holder shares a block, dec_ref when it lets go, the block returns to
 * the back of the free deque at zero), §3.1 (copy-on-write + ref_count), and
 * "vLLM PagedAttention source notes" §2.1 (allocate / free / append_slot) and
 * §3 (fragmentation ratio).
 *
 * Sequences are identified by caller ids (int64).  A sequence's table always
 * spans exactly ceil((offset + num_tokens) / block_size) blocks.  Appending
 * fills the last block, then takes fresh blocks in deque order.  If the
 * block the first appended token lands in is shared (ref_count > 1), it is
 * first replaced in this sequence by a fresh block (copy-on-write) and the
 * pair (shared, fresh) is returned for the caller to copy on the device
 * (pkv_copy_blocks).  Every failing call leaves the allocator unchanged.
 * ------------------------------------------------------------------------ */
typedef struct pkv_allocator pkv_allocator;

/* free_order: NULL for ids 0..num_blocks-1 in order, else a host permutation
 * of them giving the initial deque order.  *out receives the allocator. */
PKV_API pkv_status pkv_alloc_create(int64_t num_blocks, int32_t block_size,
                                    const int32_t* free_order, pkv_allocator** out);
PKV_API pkv_status pkv_alloc_destroy(pkv_allocator* a);
/* Number of free blocks; -1 for a null allocator. */
PKV_API int64_t pkv_alloc_num_free(const pkv_allocator* a);
/* ref_count of a block (0 = free); -1 for a bad block id. */
PKV_API int32_t pkv_alloc_ref_count(const pkv_allocator* a, int64_t block);
/* Take n blocks from the front of the deque into out_ids (host, n entries),
 * each with ref_count 1; PKV_ERR_NO_BLOCKS if fewer than n are free. */
PKV_API pkv_status pkv_alloc_blocks(pkv_allocator* a, int64_t n, int32_t* out_ids);
PKV_API pkv_status pkv_alloc_inc_ref(pkv_allocator* a, int32_t block);
/* At zero the block goes to the back of the deque.  A free block: error. */
PKV_API pkv_status pkv_alloc_dec_ref(pkv_allocator* a, int32_t block);

/* New empty sequence whose first token will sit at row `offset` of its first
 * block (0 <= offset < block_size). */
PKV_API pkv_status pkv_seq_new(pkv_allocator* a, int64_t seq_id, int32_t offset);
/* Prefix hit: an empty sequence takes n already allocated blocks (inc_ref
 * each) covering num_tokens tokens; n must equal
 * ceil((offset + num_tokens) / block_size). */
PKV_API pkv_status pkv_seq_share(pkv_allocator* a, int64_t seq_id, const int32_t* blocks,
                                 int32_t n, int64_t num_tokens);
/* Append num_tokens tokens.  slots_out (nullable, num_tokens entries)
 * receives their slots (block * block_size + row).  cow_src / cow_dst
 * (nullable, one entry each) and *n_cow (nullable) receive the copy-on-write
 * pair, if any (n_cow is 0 or 1).  PKV_ERR_NO_BLOCKS: nothing changed. */
PKV_API pkv_status pkv_seq_append(pkv_allocator* a, int64_t seq_id, int64_t num_tokens,
                                  int64_t* slots_out, int32_t* cow_src, int32_t* cow_dst,
                                  int32_t* n_cow);
/* One decode step for many sequences: for i < n, append num_tokens[i]
 * tokens (NULL: one each) to seq_ids[i], in order, as pkv_seq_append would.
 * slots_out (nullable) receives every appended token's slot, sequence by
 * sequence (the step's slot_mapping); cow_src / cow_dst (nullable, room for n
 * entries) and *n_cow receive the copy-on-write pairs.  All or nothing: if
 * the blocks the whole batch needs (copy-on-write included, in order) are
 * not free, PKV_ERR_NO_BLOCKS and nothing changes; an unknown id or a repeated
 * id is PKV_ERR_INVALID_ARG. */
PKV_API pkv_status pkv_seq_append_batch(pkv_allocator* a, const int64_t* seq_ids, int32_t n,
                                        const int64_t* num_tokens, int64_t* slots_out,
                                        int32_t* cow_src, int32_t* cow_dst, int32_t* n_cow);

/* dst (new id) shares every block of src (inc_ref each), same offset and
 * length. */
PKV_API pkv_status pkv_seq_fork(pkv_allocator* a, int64_t src, int64_t dst);
/* Release every block of the sequence (dec_ref) and forget it. */
PKV_API pkv_status pkv_seq_free(pkv_allocator* a, int64_t seq_id);
PKV_API pkv_status pkv_seq_info(const pkv_allocator* a, int64_t seq_id, int64_t* num_tokens,
                                int32_t* offset, int32_t* num_blocks);
/* Host arrays for the kernels: tables [batch, max_blocks] (row b = blocks of
 * seq_ids[b], padded with -1), seq_lens [batch], offsets [batch] (both
 * nullable).  PKV_ERR_CAPACITY if a sequence spans more than max_blocks. */
PKV_API pkv_status pkv_seq_tables(const pkv_allocator* a, const int64_t* seq_ids, int32_t batch,
                                  int32_t max_blocks, int32_t* tables, int32_t* seq_lens,
                                  int32_t* offsets);
/* Allocated blocks (ref_count > 0), used slots (rows holding a token of some
 * sequence, each counted once) and the fragmentation ratio
 * (allocated * block_size - used) / (allocated * block_size), 0 when nothing
 * is allocated ("vLLM PagedAttention source notes" §3).  Any output may be
 * NULL. */
PKV_API pkv_status pkv_alloc_stats(const pkv_allocator* a, int64_t* allocated_blocks,
                                   int64_t* used_slots, double* fragmentation);

/* Static description of a status code. */
PKV_API const char* pkv_status_string(pkv_status status);

/* Library version, major * 10000 + minor * 100 + patch. */
PKV_API int32_t pkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
