// pkv_host.cu -- host-side parts of the C ABI: version, device error word, validation of
// host copies of block tables and slot mappings, the RoPE table, and per-device lookups.
#include <cmath>
#include <mutex>
#include <unordered_set>

#include "pkv_internal.h"

namespace {

// Bounds guards in the kernels OR their PKV_DEVERR_* bits in here; the host reads it back
// with pkv_device_error().
__device__ unsigned int g_device_error;

constexpr int kMaxDevices = 64;

int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}

}  // namespace

namespace pkv {

unsigned int* device_error_ptr() {
  static std::mutex mu;
  static unsigned int* ptrs[kMaxDevices] = {};
  const int dev = current_device();
  if (dev < 0) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<unsigned int*>(p);
  }
  return ptrs[dev];
}

int sm_count() {
  static std::mutex mu;
  static int counts[kMaxDevices] = {};
  const int dev = current_device();
  if (dev < 0) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (!counts[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    counts[dev] = n;
  }
  return counts[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, []() {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

}  // namespace pkv

extern "C" {

int pkv_version(void) { return 100; }  // 0.1.0

int pkv_device_error(unsigned int* err_out, int clear, pkv_stream_t stream) {
  if (!err_out) return PKV_EINVAL;
  unsigned int* dptr = pkv::device_error_ptr();
  if (!dptr) return pkv::cuda_status(cudaGetLastError());
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned int host = 0;
  cudaError_t e = cudaMemcpyAsync(&host, dptr, sizeof(host), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess && clear) e = cudaMemsetAsync(dptr, 0, sizeof(unsigned int), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return pkv::cuda_status(e);
  *err_out = host;
  return PKV_OK;
}

int pkv_rope_table(float* cos_sin, int n_index, int head_dim, double base) {
  if (!cos_sin || n_index <= 0 || head_dim <= 0 || (head_dim & 1) || !(base > 0.0))
    return PKV_EINVAL;
  const int half = head_dim / 2;
  for (int j = 0; j < n_index; ++j) {
    for (int i = 0; i < half; ++i) {
      const double inv_freq = std::pow(base, -2.0 * static_cast<double>(i) / head_dim);
      const double ang = static_cast<double>(j) * inv_freq;
      cos_sin[(static_cast<size_t>(j) * half + i) * 2 + 0] = static_cast<float>(std::cos(ang));
      cos_sin[(static_cast<size_t>(j) * half + i) * 2 + 1] = static_cast<float>(std::sin(ang));
    }
  }
  return PKV_OK;
}

int pkv_check_tables(const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                     int max_blocks_per_seq, int block_size, int num_blocks, int* bad_seq) {
  if (num_seqs < 0 || max_blocks_per_seq < 0 || block_size <= 0 || num_blocks < 0)
    return PKV_EINVAL;
  if (num_seqs > 0 && (!block_tables || !context_lens)) return PKV_EINVAL;
  const int64_t cap = static_cast<int64_t>(max_blocks_per_seq) * block_size;
  for (int b = 0; b < num_seqs; ++b) {
    const int64_t ctx = context_lens[b];
    bool ok = ctx >= 0 && ctx <= cap;
    if (ok) {
      const int64_t nblk = (ctx + block_size - 1) / block_size;
      for (int64_t j = 0; j < nblk && ok; ++j) {
        const int32_t id = block_tables[static_cast<int64_t>(b) * max_blocks_per_seq + j];
        ok = id >= 0 && id < num_blocks;
      }
    }
    if (!ok) {
      if (bad_seq) *bad_seq = b;
      return PKV_ERANGE;
    }
  }
  return PKV_OK;
}

int pkv_check_slots(const int64_t* slots, int n, int num_blocks, int block_size, int* bad_index) {
  if (n < 0 || num_blocks < 0 || block_size <= 0 || (n > 0 && !slots)) return PKV_EINVAL;
  const int64_t limit = static_cast<int64_t>(num_blocks) * block_size;
  std::unordered_set<int64_t> seen;
  seen.reserve(static_cast<size_t>(n) * 2);
  for (int i = 0; i < n; ++i) {
    const int64_t s = slots[i];
    if (s < 0) continue;
    if (s >= limit || !seen.insert(s).second) {
      if (bad_index) *bad_index = i;
      return PKV_ERANGE;
    }
  }
  return PKV_OK;
}

}  // extern "C"
