// pkv_cache.cu -- cache-editing kernels: paged and sink+ring slot mapping, KV append
// (slot scatter) and the copy-on-write block copy.
//
// All of them move whole 16-byte vectors; a K/V row of head_dim fp16 values is head_dim / 8
// vectors, so consecutive threads cover consecutive bytes of a row (coalesced).
#include <cuda_fp16.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kThreads = 256;

// slot = table[seq][pos / bs] * bs + pos % bs  ([EDGE] addressing section).
__global__ void slot_mapping_kernel(const int32_t* __restrict__ seq_ids,
                                    const int64_t* __restrict__ positions, int n,
                                    const int32_t* __restrict__ block_tables, int num_seqs,
                                    int max_blocks, int block_size, int64_t* __restrict__ out,
                                    unsigned int* err) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int64_t p = positions[i];
  const int32_t s = seq_ids[i];
  int64_t slot = -1;
  if (p >= 0) {
    if (s < 0 || s >= num_seqs) {
      atomicOr(err, PKV_DEVERR_SEQ);
    } else if (p / block_size >= max_blocks) {
      atomicOr(err, PKV_DEVERR_POSITION);
    } else {
      const int64_t phys = block_tables[static_cast<int64_t>(s) * max_blocks + p / block_size];
      slot = phys * block_size + p % block_size;
    }
  }
  out[i] = slot;
}

// Ring slot r = Slot(pos) ([RING] §环形上下文与注意力沉淀机制), then the paged address of r.
__global__ void ring_slot_mapping_kernel(const int32_t* __restrict__ seq_ids,
                                         const int64_t* __restrict__ positions, int n,
                                         const int32_t* __restrict__ block_tables, int num_seqs,
                                         int max_blocks, int sink, int window, int block_size,
                                         int64_t* __restrict__ out, unsigned int* err) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int64_t p = positions[i];
  const int32_t s = seq_ids[i];
  int64_t slot = -1;
  if (p >= 0) {
    const int64_t r = p < sink ? p : sink + (p - sink) % window;
    if (s < 0 || s >= num_seqs) {
      atomicOr(err, PKV_DEVERR_SEQ);
    } else if (r / block_size >= max_blocks) {
      atomicOr(err, PKV_DEVERR_POSITION);
    } else {
      const int64_t phys = block_tables[static_cast<int64_t>(s) * max_blocks + r / block_size];
      slot = phys * block_size + r % block_size;
    }
  }
  out[i] = slot;
}

// One thread per 16-byte vector of one (token, K|V, kv head) row.
__global__ void kv_append_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                 const int64_t* __restrict__ slots, int num_tokens,
                                 uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                                 int64_t num_slots, int num_kv_heads, int vecs_per_row,
                                 int block_size, unsigned int* err) {
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t per_token = static_cast<int64_t>(2) * num_kv_heads * vecs_per_row;
  if (idx >= per_token * num_tokens) return;
  const int t = static_cast<int>(idx / per_token);
  int64_t rem = idx - t * per_token;
  const int which = static_cast<int>(rem / (static_cast<int64_t>(num_kv_heads) * vecs_per_row));
  rem -= static_cast<int64_t>(which) * num_kv_heads * vecs_per_row;
  const int h = static_cast<int>(rem / vecs_per_row);
  const int c = static_cast<int>(rem % vecs_per_row);
  const int64_t slot = slots[t];
  if (slot < 0) return;
  if (slot >= num_slots) {
    if (c == 0 && which == 0 && h == 0) atomicOr(err, PKV_DEVERR_SLOT);
    return;
  }
  const int64_t blk = slot / block_size, off = slot % block_size;
  const int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * vecs_per_row + c;
  const int64_t src = (static_cast<int64_t>(t) * num_kv_heads + h) * vecs_per_row + c;
  if (which == 0)
    k_cache[dst] = __ldg(k + src);
  else
    v_cache[dst] = __ldg(v + src);
}

// FP8 append: thread = 8 consecutive elements of one (token, K|V, kv head) row: 16 fp16 bytes
// in, each divided by the head's scale in binary32 and rounded to E4M3, 8 bytes out.
__global__ void kv_append_fp8_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                     const int64_t* __restrict__ slots, int num_tokens,
                                     uint2* __restrict__ k_cache, uint2* __restrict__ v_cache,
                                     int64_t num_slots, int num_kv_heads, int vecs_per_row,
                                     int block_size, const float* __restrict__ k_scale,
                                     const float* __restrict__ v_scale, unsigned int* err) {
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t per_token = static_cast<int64_t>(2) * num_kv_heads * vecs_per_row;
  if (idx >= per_token * num_tokens) return;
  const int t = static_cast<int>(idx / per_token);
  int64_t rem = idx - t * per_token;
  const int which = static_cast<int>(rem / (static_cast<int64_t>(num_kv_heads) * vecs_per_row));
  rem -= static_cast<int64_t>(which) * num_kv_heads * vecs_per_row;
  const int h = static_cast<int>(rem / vecs_per_row);
  const int c = static_cast<int>(rem % vecs_per_row);
  const int64_t slot = slots[t];
  if (slot < 0) return;
  if (slot >= num_slots) {
    if (c == 0 && which == 0 && h == 0) atomicOr(err, PKV_DEVERR_SLOT);
    return;
  }
  const int64_t blk = slot / block_size, off = slot % block_size;
  const int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * vecs_per_row + c;
  const int64_t src = (static_cast<int64_t>(t) * num_kv_heads + h) * vecs_per_row + c;
  const uint4 x = __ldg((which ? v : k) + src);
  const float sc = __ldg((which ? v_scale : k_scale) + h);
  (which ? v_cache : k_cache)[dst] =
      make_uint2(f16x4_to_e4m3x4(x.x, x.y, sc), f16x4_to_e4m3x4(x.z, x.w, sc));
}

// grid.y enumerates (layer, pair, K|V); grid.x strides over the block's 16-byte vectors.
__global__ void copy_blocks_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                                   const int32_t* __restrict__ src, const int32_t* __restrict__ dst,
                                   int n, int64_t layer_stride_vecs, int num_blocks,
                                   int64_t block_vecs, unsigned int* err) {
  const int job = blockIdx.y;
  const int which = job & 1;
  const int pair = (job >> 1) % n;
  const int layer = (job >> 1) / n;
  const int32_t s = src[pair], d = dst[pair];
  if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(err, PKV_DEVERR_BLOCK_ID);
    return;
  }
  uint4* base = (which ? v_cache : k_cache) + layer * layer_stride_vecs;
  const uint4* from = base + static_cast<int64_t>(s) * block_vecs;
  uint4* to = base + static_cast<int64_t>(d) * block_vecs;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < block_vecs;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    to[i] = from[i];
}

int launch_status() { return cuda_status(cudaGetLastError()); }

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" {

int pkv_slot_mapping(const int32_t* seq_ids, const int64_t* positions, int n,
                     const int32_t* block_tables, int num_seqs, int max_blocks_per_seq,
                     int block_size, int64_t* slot_out, pkv_stream_t stream) {
  if (n < 0 || num_seqs < 0 || max_blocks_per_seq < 0 || block_size <= 0) return PKV_EINVAL;
  if (n == 0) return PKV_OK;
  if (!seq_ids || !positions || !slot_out || (num_seqs > 0 && !block_tables)) return PKV_EINVAL;
  unsigned int* err = device_error_ptr();
  if (!err) return launch_status();
  slot_mapping_kernel<<<(n + kThreads - 1) / kThreads, kThreads, 0,
                        static_cast<cudaStream_t>(stream)>>>(
      seq_ids, positions, n, block_tables, num_seqs, max_blocks_per_seq, block_size, slot_out,
      err);
  return launch_status();
}

int pkv_ring_slot_mapping(const int32_t* seq_ids, const int64_t* positions, int n,
                          const int32_t* block_tables, int num_seqs, int max_blocks_per_seq,
                          int sink, int window, int block_size, int64_t* slot_out,
                          pkv_stream_t stream) {
  if (n < 0 || num_seqs < 0 || max_blocks_per_seq < 0 || block_size <= 0 || sink < 0 ||
      window < 1)
    return PKV_EINVAL;
  if (n == 0) return PKV_OK;
  if (!seq_ids || !positions || !slot_out || (num_seqs > 0 && !block_tables)) return PKV_EINVAL;
  unsigned int* err = device_error_ptr();
  if (!err) return launch_status();
  ring_slot_mapping_kernel<<<(n + kThreads - 1) / kThreads, kThreads, 0,
                             static_cast<cudaStream_t>(stream)>>>(
      seq_ids, positions, n, block_tables, num_seqs, max_blocks_per_seq, sink, window,
      block_size, slot_out, err);
  return launch_status();
}

int pkv_kv_append(const void* k, const void* v, const int64_t* slot_mapping, int num_tokens,
                  void* k_cache, void* v_cache, int num_blocks, int num_kv_heads, int head_dim,
                  int block_size, pkv_stream_t stream) {
  if (num_tokens < 0 || num_blocks < 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      head_dim % 8 != 0 || !valid_block_size(block_size))
    return PKV_EINVAL;
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PKV_EINVAL;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_EINVAL;
  unsigned int* err = device_error_ptr();
  if (!err) return launch_status();
  const int vecs = head_dim / 8;
  const int64_t total = static_cast<int64_t>(num_tokens) * 2 * num_kv_heads * vecs;
  const int64_t blocks = (total + kThreads - 1) / kThreads;
  if (blocks > 0x7fffffff) return PKV_EINVAL;
  kv_append_kernel<<<static_cast<unsigned>(blocks), kThreads, 0,
                     static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(k), static_cast<const uint4*>(v), slot_mapping, num_tokens,
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache),
      static_cast<int64_t>(num_blocks) * block_size, num_kv_heads, vecs, block_size, err);
  return launch_status();
}

int pkv_kv_append_fp8(const void* k, const void* v, const int64_t* slot_mapping, int num_tokens,
                      void* k_cache, void* v_cache, int num_blocks, int num_kv_heads,
                      int head_dim, int block_size, const float* k_scale, const float* v_scale,
                      pkv_stream_t stream) {
  if (num_tokens < 0 || num_blocks < 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      head_dim % 8 != 0 || !valid_block_size(block_size))
    return PKV_EINVAL;
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache || !k_scale || !v_scale)
    return PKV_EINVAL;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_EINVAL;
  unsigned int* err = device_error_ptr();
  if (!err) return launch_status();
  const int vecs = head_dim / 8;
  const int64_t total = static_cast<int64_t>(num_tokens) * 2 * num_kv_heads * vecs;
  const int64_t blocks = (total + kThreads - 1) / kThreads;
  if (blocks > 0x7fffffff) return PKV_EINVAL;
  kv_append_fp8_kernel<<<static_cast<unsigned>(blocks), kThreads, 0,
                         static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(k), static_cast<const uint4*>(v), slot_mapping, num_tokens,
      static_cast<uint2*>(k_cache), static_cast<uint2*>(v_cache),
      static_cast<int64_t>(num_blocks) * block_size, num_kv_heads, vecs, block_size, k_scale,
      v_scale, err);
  return launch_status();
}

int pkv_copy_blocks(void* k_cache, void* v_cache, const int32_t* src, const int32_t* dst, int n,
                    int64_t layer_stride_elems, int num_layers, int num_blocks,
                    int num_kv_heads, int head_dim, int block_size, pkv_stream_t stream) {
  if (n < 0 || num_layers < 0 || num_blocks < 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      head_dim % 8 != 0 || !valid_block_size(block_size) || layer_stride_elems < 0 ||
      layer_stride_elems % 8 != 0)
    return PKV_EINVAL;
  if (n == 0 || num_layers == 0) return PKV_OK;
  if (!k_cache || !v_cache || !src || !dst) return PKV_EINVAL;
  if (!aligned16(k_cache) || !aligned16(v_cache)) return PKV_EINVAL;
  const int64_t block_elems = static_cast<int64_t>(num_kv_heads) * block_size * head_dim;
  if (num_layers > 1 && layer_stride_elems < block_elems * num_blocks) return PKV_EINVAL;
  const int64_t jobs = static_cast<int64_t>(n) * num_layers * 2;
  if (jobs > 65535) return PKV_EINVAL;
  unsigned int* err = device_error_ptr();
  if (!err) return launch_status();
  const int64_t block_vecs = block_elems / 8;
  const int64_t per_cta = kThreads * 4;
  const unsigned gx = static_cast<unsigned>(std::min<int64_t>((block_vecs + per_cta - 1) / per_cta, 1024));
  dim3 grid(gx, static_cast<unsigned>(jobs));
  copy_blocks_kernel<<<grid, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), src, dst, n,
      layer_stride_elems / 8, num_blocks, block_vecs, err);
  return launch_status();
}

}  // extern "C"
