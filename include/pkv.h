/*
 * pkv.h -- C ABI of the paged KV-cache decode-attention library (GB300, sm_103a).
 *
 * The operations are the hot path of a paged KV cache:
 *   - slot mapping: a token's logical position -> its slot in the physical block pool, through
 *     the sequence's block table (and the sink + ring variant of that mapping);
 *   - KV append: scatter each new token's K/V rows into its slot;
 *   - copy-on-write block copy;
 *   - paged decode attention: each sequence's few newest query tokens attend over all of its
 *     cached K/V, read indirectly through its block table, with GQA head groups;
 *   - sink + ring decode attention with RoPE applied at read time;
 * and around it: an FP8 (E4M3) form of the cache with its append and decode, verification of
 * speculative drafts (accept/reject, next token), and a host block pool that hands out the
 * block tables (prefix sharing, reference counts, copy-on-write pairs).
 *
 * Sources (page title, section):
 *   [EDGE]   "端侧 SLM 显存保活术：在 4GB 内存板卡上实现轻量 PagedAttention 与 KV 缓存分块"
 *   [OLLAMA] "Ollama的内存管理策略：从KV Cache Block分配到Prefix-aware内存复用的演进"
 *   [RING]   streaming-inference page (wzjinhao.cn/news/69573), sections
 *            "环形上下文与注意力沉淀机制" and "C 环形 KV 缓存管理内核实现"
 *   [VLLM]   "大模型推理内存优化：从 KV Cache 分页到连续批处理的工程实践"
 *
 * Conventions shared by every entry point
 *   - Pointers marked (device) are CUDA device pointers; (host) are host pointers. The caller
 *     owns every buffer. Nothing here allocates device memory or synchronises the stream,
 *     except pkv_device_error(), which reads a status word back (the host block pool
 *     allocates its own host bookkeeping).
 *   - fp16 tensors are IEEE binary16 ("half"), passed as void*.
 *   - One layer's KV pool: k_cache and v_cache, each [num_blocks][num_kv_heads][block_size]
 *     [head_dim] contiguous, 16-byte aligned. Several layers are addressed by the caller
 *     passing each layer's base pointer.
 *   - head_dim must be 128. block_size must be one of 16, 32, 64, 128, 256.
 *   - GQA: query head h reads kv head h / (num_q_heads / num_kv_heads).
 *   - Block tables: int32 [num_seqs][max_blocks_per_seq]; entry j of row b is the physical
 *     block holding logical block j of sequence b ([EDGE] §注意力寻址非连续物理块的间接寻址内核;
 *     [VLLM] block-table list). Entries past a sequence's last block are never read.
 *   - Return value: PKV_OK (0) or a negative status. Argument errors are detected on the host
 *     before any launch. Data-dependent errors found on the device (an out-of-range block id
 *     or context length) never fault: the kernel skips the bad access and sets a bit in the
 *     device error word (see pkv_device_error).
 *   - stream: a cudaStream_t (NULL = the legacy default stream).
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef void* pkv_stream_t;

/* ---- status codes ------------------------------------------------------------------------ */
#define PKV_OK 0
#define PKV_EINVAL (-22)      /* bad shape, size, alignment or pointer */
#define PKV_ERANGE (-34)      /* a host-checked index is out of range (pkv_check_*) */
#define PKV_ENOSPC (-28)      /* workspace (or the fixed scratch array) too small for the call */
#define PKV_ECUDA_BASE (-1000) /* PKV_ECUDA_BASE - cudaError_t of a failed CUDA call */

/* ---- device error word bits ---------------------------------------------------------------- */
#define PKV_DEVERR_BLOCK_ID 1u   /* a block-table entry outside [0, num_blocks) was read */
#define PKV_DEVERR_CONTEXT 2u    /* a context length outside [0, max_blocks*block_size] */
#define PKV_DEVERR_SLOT 4u       /* a slot outside [-inf, num_blocks*block_size) (negative = skip) */
#define PKV_DEVERR_TIMEOUT 8u    /* an in-kernel pipeline wait ran past its iteration limit */
#define PKV_DEVERR_SEQ 16u       /* a sequence id outside [0, num_seqs) */
#define PKV_DEVERR_POSITION 32u  /* a position past the sequence's block table */
#define PKV_DEVERR_TOKEN 64u     /* a draft token id outside [0, vocab) (treated as rejected) */

/* Library version (major*10000 + minor*100 + patch). */
int pkv_version(void);

/* Reads the calling device's error word into *err_out (host) after synchronising `stream`;
 * clears it when `clear` is non-zero. Bits: PKV_DEVERR_*. */
int pkv_device_error(unsigned int* err_out, int clear, pkv_stream_t stream);

/* ---- slot mapping ------------------------------------------------------------------------
 * slot_out[i] = block_tables[seq_ids[i]][positions[i] / block_size] * block_size
 *               + positions[i] % block_size,
 * the addressing of [EDGE] §注意力寻址非连续物理块的间接寻址内核 (logical block = T / block size,
 * offset = T % block size, physical block from the table). positions[i] < 0 gives -1
 * (padding). A seq id or position outside the table gives -1 and sets PKV_DEVERR_SEQ /
 * PKV_DEVERR_POSITION. All arrays (device): seq_ids int32 [n], positions int64 [n],
 * slot_out int64 [n]. */
int pkv_slot_mapping(const int32_t* seq_ids, const int64_t* positions, int n,
                     const int32_t* block_tables, int num_seqs, int max_blocks_per_seq,
                     int block_size, int64_t* slot_out, pkv_stream_t stream);

/* Sink + ring slot mapping ([RING] §环形上下文与注意力沉淀机制): ring slot
 *   r = positions[i]               if positions[i] < sink
 *     = sink + (positions[i] - sink) mod window   otherwise,
 * then slot = block_tables[seq][r / block_size] * block_size + r % block_size. The ring's
 * sink + window slots occupy the first ceil((sink+window)/block_size) table entries.
 * Arrays as for pkv_slot_mapping. window >= 1, sink >= 0. */
int pkv_ring_slot_mapping(const int32_t* seq_ids, const int64_t* positions, int n,
                          const int32_t* block_tables, int num_seqs, int max_blocks_per_seq,
                          int sink, int window, int block_size, int64_t* slot_out,
                          pkv_stream_t stream);

/* ---- KV append ---------------------------------------------------------------------------
 * For every token t with slot_mapping[t] >= 0 and every kv head h:
 *   k_cache[slot / bs][h][slot % bs][:] = k[t][h][:]   (and the same for v),
 * a byte copy ([VLLM] on-demand paging: a new token's K/V go into its block; [RING] AppendKV).
 * Negative slots are skipped. A slot >= num_blocks*block_size is skipped and sets
 * PKV_DEVERR_SLOT. k, v (device): fp16 [num_tokens][num_kv_heads][head_dim];
 * slot_mapping (device): int64 [num_tokens]. Duplicate slots in one call race. */
int pkv_kv_append(const void* k, const void* v, const int64_t* slot_mapping, int num_tokens,
                  void* k_cache, void* v_cache, int num_blocks, int num_kv_heads, int head_dim,
                  int block_size, pkv_stream_t stream);

/* ---- copy-on-write block copy --------------------------------------------------------------
 * For every layer l < num_layers and i < n: block dst[i] := block src[i], K and V, where
 * layer l's pool starts layer_stride_elems fp16 elements after layer l-1's and a block is
 * num_kv_heads*block_size*head_dim elements ([OLLAMA] §三, copy-on-write of a shared block
 * before a write). src, dst (device): int32 [n]; ids outside [0, num_blocks) are skipped and
 * set PKV_DEVERR_BLOCK_ID. The dst set must not overlap the src set. */
int pkv_copy_blocks(void* k_cache, void* v_cache, const int32_t* src, const int32_t* dst, int n,
                    int64_t layer_stride_elems, int num_layers, int num_blocks,
                    int num_kv_heads, int head_dim, int block_size, pkv_stream_t stream);

/* ---- decode attention ------------------------------------------------------------------------
 * Workspace: caller-owned device scratch for split-context partial results and the per
 * (sequence, kv head) arrival counters. Size it with pkv_decode_workspace_bytes() (for the
 * current device; the size depends on its SM count) and zero it once with
 * pkv_workspace_init() before first use; every decode call leaves the counters zeroed again.
 * One workspace must not be used by two calls that run concurrently. After a call that set
 * PKV_DEVERR_TIMEOUT, re-initialise it. */
size_t pkv_decode_workspace_bytes(int num_seqs, int q_len, int num_q_heads, int num_kv_heads,
                                  int head_dim);

/* Turns the launch overlap of the fused-append calls (pkv_paged_attn_decode_append, its FP8
 * form and pkv_ring_attn_decode_append) on (enable != 0, the default) or off, for every call made afterwards in this process,
 * including calls captured into a CUDA graph afterwards. With it off a fused call starts only
 * after the kernel before it has completed, so it may follow a kernel that writes its pools,
 * block tables or context lengths. Returns the previous setting (0 or 1). Not part of the
 * pages' design: a scheduling control of this implementation. */
int pkv_set_early_start(int enable);
int pkv_workspace_init(void* workspace, size_t workspace_bytes, pkv_stream_t stream);

/* Paged decode attention ([VLLM] PagedAttention kernel paragraph: K/V read indirectly through
 * the block table; [EDGE] addressing section). For sequence b, query token i < q_len, query
 * head h (kv head kh = h / G):
 *   visible tokens  t < context_lens[b] - q_len + i + 1   (causal when q_len > 1)
 *   K_t = k_cache[block_tables[b][t / bs]][kh][t % bs][:]  (V likewise)
 *   out[b][i][h][:] = softmax_t(scale * <q[b][i][h], K_t>) . V
 * context_lens (device, int32 [num_seqs]) count the tokens in cache including this step's
 * appended ones. q, out (device): fp16 [num_seqs][q_len][num_q_heads][head_dim]. fp32
 * accumulation; the result is bit-identical for identical inputs and does not depend on which
 * physical blocks hold the data. A sequence with no visible tokens gets zeros. Requires
 * num_q_heads % num_kv_heads == 0 and (num_q_heads / num_kv_heads) * q_len <= 32. */
int pkv_paged_attn_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                          int num_blocks, const int32_t* block_tables, int max_blocks_per_seq,
                          const int32_t* context_lens, int num_seqs, int q_len, int num_q_heads,
                          int num_kv_heads, int head_dim, int block_size, float scale,
                          void* workspace, size_t workspace_bytes, pkv_stream_t stream);

/* Decode step with the KV append fused in: for every sequence b and new token i < q_len, the
 * token at position p = context_lens[b] - q_len + i (p >= 0) has its K/V rows k_new, v_new
 * [(b * q_len + i)][kh][:] written to the slot the block table maps p to (the slot of
 * pkv_slot_mapping), exactly as pkv_kv_append would; the attention of pkv_paged_attn_decode then
 * runs over the cache including them ([VLLM] on-demand paging + PagedAttention kernel
 * paragraph). One launch instead of slot mapping + append + decode; the new rows are read once
 * and used both for the pool and for this step's attention. k_new, v_new (device): fp16
 * [num_seqs * q_len][num_kv_heads][head_dim]; other arguments as for pkv_paged_attn_decode. The
 * slots written must not be shared with another sequence (copy-on-write first).
 * Launch overlap: by default this call is launched with programmatic dependent launch, so it
 * may start while the kernel before it on the stream is still finishing. Before that kernel
 * completes it reads only the K/V pools, block_tables and context_lens; q, k_new, v_new, out and
 * the workspace are touched after. Those three inputs must therefore not be written by the
 * immediately preceding kernel: not by a preceding pkv_paged_attn_decode_append on the same
 * pools, not by pkv_copy_blocks, and not by the caller's own kernel (say, one that advances
 * context_lens on the device). A copy (cudaMemcpyAsync) or any other kernel in between is
 * enough; otherwise turn the overlap off with pkv_set_early_start(0). The library's other
 * kernels never let the next kernel start early. */
int pkv_paged_attn_decode_append(void* out, const void* q, const void* k_new, const void* v_new,
                                 void* k_cache, void* v_cache, int num_blocks,
                                 const int32_t* block_tables, int max_blocks_per_seq,
                                 const int32_t* context_lens, int num_seqs, int q_len,
                                 int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                 float scale, void* workspace, size_t workspace_bytes,
                                 pkv_stream_t stream);

/* Chunked-prefill paged attention ([VLLM] §工程权衡, chunked prefill: a long prompt is processed
 * in chunks, each attending over the paged cache that already holds the earlier chunks). The
 * operation is pkv_paged_attn_decode's with a long query chunk: for sequence b, chunk token
 * i < q_len at position p = context_lens[b] - q_len + i and query head h (kv head h / G),
 *   out[b][i][h][:] = softmax_t(scale * <q[b][i][h], K_t>) . V,   t <= p   (causal),
 * with K_t, V_t read through the block table. context_lens count the tokens in cache including
 * the chunk, whose K/V rows must already be in the pools (pkv_kv_append first). A query with no
 * visible token (p < 0) gets zeros. q, out (device): fp16 [num_seqs][q_len][num_q_heads]
 * [head_dim]; caches, tables and lengths as for pkv_paged_attn_decode. Runs on the tensor
 * cores (tcgen05, f16 operands, f32 accumulation); needs no workspace. Requires
 * num_q_heads / num_kv_heads <= 128. The result is bit-identical for identical inputs and does
 * not depend on which physical blocks hold the data. */
int pkv_paged_prefill(void* out, const void* q, const void* k_cache, const void* v_cache,
                      int num_blocks, const int32_t* block_tables, int max_blocks_per_seq,
                      const int32_t* context_lens, int num_seqs, int q_len, int num_q_heads,
                      int num_kv_heads, int head_dim, int block_size, float scale,
                      pkv_stream_t stream);

/* Paged decode attention for callers that cannot allocate device memory: the same operation,
 * arguments and result as pkv_paged_attn_decode, with the scratch (arrival counters and
 * split-context partials) taken from a fixed array inside the library instead of a caller
 * workspace. Meant for code that runs where it may not allocate: under a host framework that
 * owns every device allocation (a plugin interface), in an embedded runtime with a fixed
 * memory budget, or at a point where entering an allocator is not allowed. The pages have no
 * counterpart of this entry point; it is an integration convenience.
 *   - The array is 8 MiB, held by every GPU that loads the library until the process exits.
 *     With R = (num_q_heads / num_kv_heads) * q_len rows per unit and S the device's SM count,
 *     a call fits if  up(4 * num_seqs * num_kv_heads) + up(8 * S * R * 16) + up(8 * S * R * 512)
 *     <= 8 MiB, where up() rounds up to a multiple of 256 (arrival counters, then the (m, l)
 *     and o[128] records of 2 partials for each of up to 4 CTAs per SM). On a 152-SM GPU that
 *     is R <= 13 (for num_seqs * num_kv_heads <= 10496). A call that does not fit returns
 *     PKV_ENOSPC and launches nothing. Shapes pkv_paged_attn_decode rejects return PKV_EINVAL,
 *     also for num_seqs == 0; a batch of 0 sequences with valid shapes returns PKV_OK.
 *   - It allocates nothing: no cudaMalloc, no cudaFree. Each call clears the arrival counters
 *     with one cudaMemsetAsync on `stream`, then launches the decode kernel.
 *   - The first call on a device resolves the array's device address (cudaGetSymbolAddress)
 *     and caches it; make that first call before any stream capture.
 *   - All calls share the one array: calls that can overlap on the GPU (different streams, or
 *     other threads) race and corrupt each other's results. Serialise them. */
int pkv_paged_attn_decode_noalloc(void* out, const void* q, const void* k_cache,
                                  const void* v_cache, int num_blocks,
                                  const int32_t* block_tables, int max_blocks_per_seq,
                                  const int32_t* context_lens, int num_seqs, int q_len,
                                  int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                  float scale, pkv_stream_t stream);

/* RoPE table for ring attention, written to HOST memory: cos_sin[j][i][0] = cos(j * theta_i),
 * cos_sin[j][i][1] = sin(j * theta_i), theta_i = base^(-2i/head_dim), j < n_index,
 * i < head_dim/2; angles computed in double, stored as float. Copy it to the device for
 * pkv_ring_attn_decode. */
int pkv_rope_table(float* cos_sin, int n_index, int head_dim, double base);

/* Sink + ring decode attention ([RING] §环形上下文与注意力沉淀机制, §C 环形 KV 缓存管理内核实现).
 * Sequence b's logical positions live at ring slots Slot(p) (see pkv_ring_slot_mapping) in
 * its first ceil((sink+window)/bs) blocks. logical_len[b] = L (tokens after this step's
 * appends), high_water[b] = hw (one past the largest position ever written), with
 * hw - window <= L <= hw. Query i (position L - q_len + i) sees the sinks [0, min(sink, vis))
 * and the window positions [max(sink, hw - window), vis), vis = L - q_len + i + 1.
 * Keys are stored before RoPE and rotated at read time (rotate-half pairs (d, d + 64)) by
 * their cache index: a sink's index is its position, a window position p has index
 * sink + p - max(sink, hw - window); the query uses its own position's index.
 * rope_cos_sin (device): float [sink + window][head_dim/2][2] from pkv_rope_table().
 * logical_len, high_water (device): int64 [num_seqs]. Other arguments as for
 * pkv_paged_attn_decode (the same workspace sizing applies). */
int pkv_ring_attn_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                         int num_blocks, const int32_t* block_tables, int max_blocks_per_seq,
                         const int64_t* logical_len, const int64_t* high_water, int num_seqs,
                         int q_len, int num_q_heads, int num_kv_heads, int head_dim,
                         int block_size, int sink, int window, const float* rope_cos_sin,
                         float scale, void* workspace, size_t workspace_bytes,
                         pkv_stream_t stream);

/* Sink + ring decode step with the KV append fused in ([RING] §C 环形 KV 缓存管理内核实现: AppendKV
 * then attention over FillValidPhysicalIndices' slots, in one launch): for every sequence b and
 * new token i < q_len at position p = logical_len[b] - q_len + i, its K/V rows k_new, v_new
 * [(b * q_len + i)][kh][:] are written (before RoPE) to ring slot Slot(p) of pkv_ring_slot_mapping,
 * exactly as pkv_ring_slot_mapping + pkv_kv_append would, and pkv_ring_attn_decode then runs
 * over the cache including them. logical_len and high_water are the values after this step's
 * appends (hw >= L). Requires q_len <= window (the new rows' slots are distinct). Launch overlap
 * as for pkv_paged_attn_decode_append: before the preceding kernel completes the call reads the
 * pools, block_tables, logical_len, high_water and rope_cos_sin, so none of them may be written
 * by the immediately preceding kernel (or call pkv_set_early_start(0)). Other arguments,
 * workspace and errors as for pkv_ring_attn_decode. */
int pkv_ring_attn_decode_append(void* out, const void* q, const void* k_new, const void* v_new,
                                void* k_cache, void* v_cache, int num_blocks,
                                const int32_t* block_tables, int max_blocks_per_seq,
                                const int64_t* logical_len, const int64_t* high_water,
                                int num_seqs, int q_len, int num_q_heads, int num_kv_heads,
                                int head_dim, int block_size, int sink, int window,
                                const float* rope_cos_sin, float scale, void* workspace,
                                size_t workspace_bytes, pkv_stream_t stream);

/* ---- FP8 (E4M3) KV cache -------------------------------------------------------------------
 * [VLLM] §工程权衡 (量化与 KV Cache 精度的权衡): FP8 halves the KV cache and is the conservative
 * choice for KV (rather than INT4). The page fixes no layout; here the pools hold E4M3 bytes
 * (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; S.1111.111 is NaN; largest finite
 * 448) in the fp16 pools' layout [num_blocks][num_kv_heads][block_size][head_dim], one byte per
 * element, and every (layer, kv head) has a K and a V scale: element value = code * scale.
 * k_scale, v_scale (device): float [num_kv_heads], positive, owned by the caller.
 *
 * pkv_kv_append_fp8: pkv_kv_append's scatter, each element stored as E4M3(x / scale[kh]): the
 * fp16 value is divided by the scale in binary32 and rounded to nearest (ties to even), finite
 * values past 448 saturate to +-448. Same slot rules and errors as pkv_kv_append; k, v fp16
 * [num_tokens][num_kv_heads][head_dim] (16-byte aligned), caches 16-byte aligned. */
int pkv_kv_append_fp8(const void* k, const void* v, const int64_t* slot_mapping, int num_tokens,
                      void* k_cache, void* v_cache, int num_blocks, int num_kv_heads,
                      int head_dim, int block_size, const float* k_scale, const float* v_scale,
                      pkv_stream_t stream);

/* pkv_paged_attn_decode over an E4M3 cache: K_t = code * k_scale[kh], V_t = code * v_scale[kh]
 * (the codes are widened to fp16 exactly, the scales applied in fp32 to the scores and the
 * output). Requires (num_q_heads / num_kv_heads) * q_len <= 8; otherwise PKV_EINVAL. Other
 * arguments, workspace and errors as for pkv_paged_attn_decode. */
int pkv_paged_attn_decode_fp8(void* out, const void* q, const void* k_cache,
                              const void* v_cache, const float* k_scale, const float* v_scale,
                              int num_blocks, const int32_t* block_tables,
                              int max_blocks_per_seq, const int32_t* context_lens, int num_seqs,
                              int q_len, int num_q_heads, int num_kv_heads, int head_dim,
                              int block_size, float scale, void* workspace,
                              size_t workspace_bytes, pkv_stream_t stream);

/* pkv_paged_attn_decode_append over an E4M3 cache: the step's new rows k_new, v_new (fp16, as for
 * pkv_paged_attn_decode_append) are stored as pkv_kv_append_fp8 stores them (the same codes) and
 * attended over as pkv_paged_attn_decode_fp8 reads the cache. One launch per layer, with the
 * early-start contract of pkv_paged_attn_decode_append (k_scale and v_scale are read after the
 * preceding kernel completes). Requires (num_q_heads / num_kv_heads) * q_len <= 8. */
int pkv_paged_attn_decode_append_fp8(void* out, const void* q, const void* k_new,
                                     const void* v_new, void* k_cache, void* v_cache,
                                     const float* k_scale, const float* v_scale, int num_blocks,
                                     const int32_t* block_tables, int max_blocks_per_seq,
                                     const int32_t* context_lens, int num_seqs, int q_len,
                                     int num_q_heads, int num_kv_heads, int head_dim,
                                     int block_size, float scale, void* workspace,
                                     size_t workspace_bytes, pkv_stream_t stream);

/* ---- speculative verification ------------------------------------------------------------
 * [RING] deferred speculative decoding: draft token x is accepted with probability
 * min(1, P_target(x) / P_draft(x)); the first rejection ends the accepted run, whose rejected
 * drafts the caller rolls back (pkv_ring_* take logical_len - rejected). With the draws given,
 * draft k of sequence b is accepted iff u_accept[b][k] * P_draft(x) < P_target(x), P the
 * softmax of the logits. n_accept[b] = the accepted run's length; next_token[b] = a draw
 * (inverse CDF: the first v whose running weight exceeds u_sample[b] x the total) from the
 * normalised residual max(0, P_target - P_draft) at the first rejected position, or from
 * P_target at position K when all K drafts are accepted.
 * target_logits float [num_seqs][num_drafts + 1][vocab], draft_logits float
 * [num_seqs][num_drafts][vocab], drafts int32 [num_seqs][num_drafts], u_accept float
 * [num_seqs][num_drafts], u_sample float [num_seqs], outputs int32 [num_seqs]; all device
 * memory; num_drafts <= 32. Each sequence is verified by a cluster of up to 8 CTAs that split
 * the vocabulary. The softmax sums are fp32 reductions: a decision on a tie within their
 * rounding may differ from an exact one. A draft id outside [0, vocab) counts as rejected and
 * sets PKV_DEVERR_TOKEN. */
int pkv_spec_verify(const float* target_logits, const float* draft_logits, const int32_t* drafts,
                    const float* u_accept, const float* u_sample, int num_seqs, int num_drafts,
                    int vocab, int32_t* n_accept, int32_t* next_token, pkv_stream_t stream);

/* ---- host block pool ------------------------------------------------------------------------
 * The host side of paging ([OLLAMA] §三 KV Cache内存管理的工程实现, and its copy-on-write
 * paragraph): num_blocks physical blocks of block_size tokens, a FIFO free list, a reference
 * count per block, and a prefix index so that sequences whose prompts begin with the same full
 * blocks of token ids share those blocks. It hands out the block tables and the copy pairs the
 * CUDA entry points take; it owns no device memory. All arrays are HOST int32; every call
 * locks the pool (one pool may serve several threads). Errors: PKV_EINVAL (bad arguments,
 * a table entry that is not a held block, an output array too small), PKV_ENOSPC (not enough
 * blocks even after reclaiming warm ones); a failed call changes nothing.
 *
 * Prefix index: full blocks only, keyed by 64-bit FNV-1a (offset basis 0xcbf29ce484222325,
 * prime 0x100000001b3, each token id xor-ed in as a 32-bit value) over the whole prefix up to
 * the block's last token (a hash chain); a candidate is reused only if its token ids and the
 * block before it match (hash_bits < 64 truncates the key, for tests of that check).
 *
 * pkv_pool_allocate: reuses the indexed blocks that match the prompt's leading full blocks
 * (reference +1; *reused of them), then takes ceil((max(max_tokens, n_tokens) - reused *
 * block_size) / block_size) blocks from the free list (reference 1) and indexes the new full
 * prompt blocks. table[0 .. *n_blocks) receives the sequence's block table.
 * pkv_pool_warm: indexes a prompt's full blocks without holding them (reference 0): they stay
 * out of the free list until reused or reclaimed.
 * pkv_pool_release: reference -1 per block; at 0 a block leaves the index and goes to the back
 * of the free list.
 * pkv_pool_fork: reference +1 per block (a child that shares the parent's table).
 * pkv_pool_append: makes room for tokens [length, length + n_new) of the sequence: a block past
 * the table is taken from the pool; a block the sequence shares with others (reference > 1) is
 * replaced by a fresh one and the pair (copy_src[i], copy_dst[i]) returned, to be copied with
 * pkv_copy_blocks before the new rows are written (copy-on-write). table / *n_blocks are
 * updated in place (capacity table_cap). With all_tokens (the sequence's token ids through
 * length + n_new) the blocks the append fills are indexed when the block before them is.
 * When the free list is short, warm blocks are reclaimed oldest allocation first; blocks a
 * sequence holds never are. */
typedef struct pkv_block_pool pkv_block_pool;
int pkv_pool_create(int num_blocks, int block_size, int hash_bits, pkv_block_pool** out);
void pkv_pool_destroy(pkv_block_pool* pool);
int pkv_pool_allocate(pkv_block_pool* pool, const int32_t* tokens, int n_tokens, int max_tokens,
                      int32_t* table, int table_cap, int* n_blocks, int* reused);
int pkv_pool_warm(pkv_block_pool* pool, const int32_t* tokens, int n_tokens);
int pkv_pool_release(pkv_block_pool* pool, const int32_t* table, int n_blocks);
int pkv_pool_fork(pkv_block_pool* pool, const int32_t* table, int n_blocks);
int pkv_pool_append(pkv_block_pool* pool, int32_t* table, int* n_blocks, int table_cap,
                    int length, int n_new, const int32_t* all_tokens, int32_t* copy_src,
                    int32_t* copy_dst, int copy_cap, int* n_copies);
/* Counts: blocks, held blocks, blocks held more than once, free-list length, warm blocks. */
int pkv_pool_stats(pkv_block_pool* pool, int* total, int* used, int* shared, int* free_blocks,
                   int* warm);
/* A block's reference count (or PKV_EINVAL). */
int pkv_pool_refcount(pkv_block_pool* pool, int block);

/* ---- host-side validation (debug mode; all arrays are HOST copies) ---------------------------
 * pkv_check_tables: every block-table entry a sequence uses (the first
 * ceil(context_lens[b]/block_size)) is in [0, num_blocks), and 0 <= context_lens[b] <=
 * max_blocks_per_seq*block_size. Returns PKV_OK or PKV_ERANGE; *bad_seq (if non-NULL) gets
 * the first offending sequence.
 * pkv_check_slots: every slot is < num_blocks*block_size and no non-negative slot repeats. */
int pkv_check_tables(const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                     int max_blocks_per_seq, int block_size, int num_blocks, int* bad_seq);
int pkv_check_slots(const int64_t* slots, int n, int num_blocks, int block_size, int* bad_index);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
