// pkv_spec.cu -- verification of speculative drafts beside the sink + ring decode: the
// streaming page's deferred speculative decoding accepts draft token x with probability
// min(1, P_target(x) / P_draft(x)), and the first rejection ends the accepted run (the
// rejected drafts are then rolled back). With the draws given, draft k is accepted iff
// u_accept * P_draft(x) < P_target(x); after a rejection at k the next token is drawn from the
// normalised residual max(0, P_target - P_draft), after K acceptances from P_target at
// position K, by inverse CDF (the first v whose running weight exceeds u_sample x total).
// One CTA per sequence; the softmax statistics and the running sums are block reductions in
// fp32, so a decision on a tie within rounding may differ from an fp64 statement.
#include <cuda_runtime.h>

#include "pkv_internal.h"

namespace {

constexpr int kSpecThreads = 1024;

__device__ __forceinline__ float block_max(float v, float* sh) {
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) sh[w] = v;
  __syncthreads();
  v = l < kSpecThreads / 32 ? sh[l] : -INFINITY;
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float block_sum(float v, float* sh) {
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) sh[w] = v;
  __syncthreads();
  v = l < kSpecThreads / 32 ? sh[l] : 0.f;
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// softmax statistics of a row: max and sum of exp(x - max)
__device__ __forceinline__ void row_stats(const float* x, int V, float* sh, float& m, float& s) {
  float mx = -INFINITY;
  for (int v = threadIdx.x; v < V; v += kSpecThreads) mx = fmaxf(mx, x[v]);
  m = block_max(mx, sh);
  float acc = 0.f;
  for (int v = threadIdx.x; v < V; v += kSpecThreads) acc += expf(x[v] - m);
  s = block_sum(acc, sh);
}

// Inverse CDF over weights w(v): the first v whose running sum exceeds u * total. Thread t owns
// the contiguous segment [t seg, (t + 1) seg); an exclusive scan of the segment sums locates
// the owner of the threshold, which walks its segment.
template <class W>
__device__ int draw(W w, int V, float u, float* sh, int* found) {
  const int seg = (V + kSpecThreads - 1) / kSpecThreads;
  const int lo = min(V, static_cast<int>(threadIdx.x) * seg), hi = min(V, lo + seg);
  float local = 0.f;
  for (int v = lo; v < hi; ++v) local += w(v);
  // scan of the per-thread sums; thread t's interval is [begin, end) with end(t) == begin(t + 1)
  // bit for bit (both are the same sums in the same order), so at most one thread owns thr
  const int wid = threadIdx.x >> 5, l = threadIdx.x & 31;
  float incl = local;
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, incl, o);
    if (l >= o) incl += y;
  }
  float prev = __shfl_up_sync(0xffffffffu, incl, 1);
  if (l == 0) prev = 0.f;
  __syncthreads();
  if (l == 31) sh[wid] = incl;
  __syncthreads();
  float warp_off = 0.f;
  for (int i = 0; i < wid; ++i) warp_off += sh[i];
  float total = warp_off;
  for (int i = wid; i < kSpecThreads / 32; ++i) total += sh[i];
  const float excl = warp_off + prev, end = warp_off + incl;
  const float thr = u * total;
  if (threadIdx.x == 0) *found = V - 1;
  __syncthreads();
  if (lo < hi && excl <= thr && thr < end) {
    float c = excl;
    int pick = hi - 1;
    for (int v = lo; v < hi; ++v) {
      c += w(v);
      if (c > thr) { pick = v; break; }
    }
    *found = pick;
  }
  __syncthreads();
  return *found;
}

__global__ void spec_verify_kernel(const float* __restrict__ tl, const float* __restrict__ dl,
                                   const int32_t* __restrict__ drafts,
                                   const float* __restrict__ ua, const float* __restrict__ us,
                                   int K, int V, int32_t* n_accept, int32_t* next_token,
                                   unsigned int* err) {
  __shared__ float sh[kSpecThreads / 32];
  __shared__ int found;
  const int b = blockIdx.x;
  int k = 0;
  for (; k < K; ++k) {
    const float* t = tl + (static_cast<int64_t>(b) * (K + 1) + k) * V;
    const float* d = dl + (static_cast<int64_t>(b) * K + k) * V;
    float mt, st, md, sd;
    row_stats(t, V, sh, mt, st);
    row_stats(d, V, sh, md, sd);
    const int x = drafts[b * K + k];
    bool accept = false;
    if (x >= 0 && x < V) {
      const float pt = expf(t[x] - mt) / st, pd = expf(d[x] - md) / sd;
      accept = ua[b * K + k] * pd < pt;
    } else if (threadIdx.x == 0) {
      atomicOr(err, PKV_DEVERR_TOKEN);
    }
    if (accept) continue;
    const int nt = draw([&](int v) {
      return fmaxf(0.f, expf(t[v] - mt) / st - expf(d[v] - md) / sd);
    }, V, us[b], sh, &found);
    if (threadIdx.x == 0) next_token[b] = nt;
    break;
  }
  if (k == K) {
    const float* t = tl + (static_cast<int64_t>(b) * (K + 1) + K) * V;
    float mt, st;
    row_stats(t, V, sh, mt, st);
    const int nt = draw([&](int v) { return expf(t[v] - mt) / st; }, V, us[b], sh, &found);
    if (threadIdx.x == 0) next_token[b] = nt;
  }
  if (threadIdx.x == 0) n_accept[b] = k;
}

}  // namespace

extern "C" int pkv_spec_verify(const float* target_logits, const float* draft_logits,
                               const int32_t* drafts, const float* u_accept,
                               const float* u_sample, int num_seqs, int num_drafts, int vocab,
                               int32_t* n_accept, int32_t* next_token, pkv_stream_t stream) {
  if (num_seqs < 0 || num_drafts < 0 || vocab < 1) return PKV_EINVAL;
  if (num_seqs == 0) return PKV_OK;
  if (!target_logits || !u_sample || !n_accept || !next_token ||
      (num_drafts > 0 && (!draft_logits || !drafts || !u_accept)))
    return PKV_EINVAL;
  unsigned int* err = pkv::device_error_ptr();
  if (!err) return pkv::cuda_status(cudaGetLastError());
  spec_verify_kernel<<<num_seqs, kSpecThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      target_logits, draft_logits, drafts, u_accept, u_sample, num_drafts, vocab, n_accept,
      next_token, err);
  return pkv::cuda_status(cudaGetLastError());
}
