// pkv_spec.cu -- verification of speculative drafts beside the sink + ring decode: the
// streaming page's deferred speculative decoding accepts draft token x with probability
// min(1, P_target(x) / P_draft(x)), and the first rejection ends the accepted run (the
// rejected drafts are then rolled back). With the draws given, draft k is accepted iff
// u_accept * P_draft(x) < P_target(x); after a rejection at k the next token is drawn from the
// normalised residual max(0, P_target - P_draft), after K acceptances from P_target at
// position K, by inverse CDF (the first v whose running weight exceeds u_sample x total).
// One thread-block cluster (up to 8 CTAs) per sequence, each CTA taking a slice of the
// vocabulary: every row's softmax statistics are online (max, sum) over the slices, combined
// through distributed shared memory; the draw scans the slices' sums. The statistics and the
// running sums are fp32 reductions, so a decision on a tie within rounding may differ from an
// fp64 statement.
#include <cuda_runtime.h>

#include <algorithm>

#include "pkv_internal.h"

namespace {

constexpr int kSpecThreads = 256;
constexpr int kMaxCluster = 8;        // CTAs per sequence (a portable cluster)
constexpr int kMaxRows = 2 * 32 + 1;  // target and draft rows of up to 32 drafts

// ---- thread-block cluster primitives (distributed shared memory) --------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}
// a float in CTA `rank`'s copy of this CTA's shared variable p
__device__ __forceinline__ float ld_cluster_f32(const float* p, uint32_t rank) {
  uint32_t local = static_cast<uint32_t>(__cvta_generic_to_shared(p)), remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

__device__ __forceinline__ float block_reduce(float v, float* sh, bool is_max) {
  for (int o = 16; o; o >>= 1) {
    const float y = __shfl_xor_sync(0xffffffffu, v, o);
    v = is_max ? fmaxf(v, y) : v + y;
  }
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) sh[w] = v;
  __syncthreads();
  v = l < kSpecThreads / 32 ? sh[l] : (is_max ? -INFINITY : 0.f);
  for (int o = 16; o; o >>= 1) {
    const float y = __shfl_xor_sync(0xffffffffu, v, o);
    v = is_max ? fmaxf(v, y) : v + y;
  }
  return v;
}

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// e^(y - m) for y <= m (0 for y = -inf), through 2^x on the scaled difference.
__device__ __forceinline__ float exp_below(float y, float m) {
  return y > -INFINITY ? fast_exp2((y - m) * kLog2e) : 0.f;
}

// Online (max, sum of exp(x - max)) over x[lo, hi), by this thread (eight independent loads in
// flight per step), then the block.
__device__ void slice_stats(const float* x, int lo, int hi, float* sh, float& m, float& s) {
  constexpr int kU = 8;
  float mx = -INFINITY, acc = 0.f;
  for (int v0 = lo + static_cast<int>(threadIdx.x); v0 < hi; v0 += kU * kSpecThreads) {
    float y[kU];
#pragma unroll
    for (int i = 0; i < kU; ++i) {
      const int v = v0 + i * kSpecThreads;
      y[i] = v < hi ? __ldg(x + v) : -INFINITY;
    }
    float bm = y[0];
#pragma unroll
    for (int i = 1; i < kU; ++i) bm = fmaxf(bm, y[i]);
    if (bm > mx) {
      acc *= exp_below(mx, bm);
      mx = bm;
    }
#pragma unroll
    for (int i = 0; i < kU; ++i) acc += exp_below(y[i], mx);
  }
  m = block_reduce(mx, sh, true);
  const float part = mx == -INFINITY ? 0.f : acc * exp_below(mx, m);
  s = block_reduce(part, sh, false);
}

// Inverse CDF over weights w(v) on this CTA's slice [lo, hi) of the cluster's vocabulary: the
// first v whose running sum exceeds u * total. Thread t owns a contiguous segment of the slice;
// a block scan of the segment sums, then a cluster scan of the slices' sums (in rank order),
// give every segment its interval [begin, end), with end == the next segment's begin bit for
// bit (the same sums in the same order), so at most one thread of the cluster owns u * total;
// if none does (rounding at the very end), the last CTA answers V - 1.
template <class W>
__device__ int draw(W w, int lo, int hi, int V, float u, float* sh, float* slice_sum,
                    int* found, uint32_t rank, int C) {
  const int n = hi - lo;
  const int seg = (n + kSpecThreads - 1) / kSpecThreads;
  const int s0 = min(hi, lo + static_cast<int>(threadIdx.x) * seg), s1 = min(hi, s0 + seg);
  float local = 0.f;
#pragma unroll 8
  for (int v = s0; v < s1; ++v) local += w(v);
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
  float warp_off = 0.f, block_total = 0.f;
  for (int i = 0; i < wid; ++i) warp_off += sh[i];
  for (int i = 0; i < kSpecThreads / 32; ++i) block_total += sh[i];
  if (threadIdx.x == 0) {
    *slice_sum = block_total;
    *found = -1;
  }
  cluster_sync();                                 // every slice's sum is published
  float slice_off = 0.f, total = 0.f;
  for (int c = 0; c < C; ++c) {
    const float t = ld_cluster_f32(slice_sum, c);
    if (c < static_cast<int>(rank)) slice_off += t;
    total += t;
  }
  const float thr = u * total;
  const float excl = slice_off + warp_off + prev, end = slice_off + warp_off + incl;
  if (s0 < s1 && excl <= thr && thr < end) {
    float c = excl;
    int pick = s1 - 1;
    for (int v = s0; v < s1; ++v) {
      c += w(v);
      if (c > thr) { pick = v; break; }
    }
    *found = pick;
  }
  // no slice owns the threshold: only rounding at the very end of the range does that
  const bool nobody = !(thr < total);
  __syncthreads();
  int res = *found;
  if (nobody && static_cast<int>(rank) == C - 1) res = V - 1;
  cluster_sync();                                 // the slice sums may be overwritten again
  return res;
}

// One cluster of C CTAs per sequence; CTA `rank` holds the vocabulary slice [rank * chunk,
// (rank + 1) * chunk). The row statistics (max, sum) are combined across the cluster in rank
// order, so every CTA takes the same decisions.
__global__ void __launch_bounds__(kSpecThreads)
spec_verify_kernel(const float* __restrict__ tl, const float* __restrict__ dl,
                   const int32_t* __restrict__ drafts, const float* __restrict__ ua,
                   const float* __restrict__ us, int K, int V, int C, int32_t* n_accept,
                   int32_t* next_token, unsigned int* err) {
  __shared__ float sh[kSpecThreads / 32];
  __shared__ float part_m[kMaxRows], part_s[kMaxRows];   // this slice's stats per row
  __shared__ float row_m[kMaxRows], row_s[kMaxRows];     // the cluster's
  __shared__ float slice_sum;
  __shared__ int found;
  const uint32_t rank = C > 1 ? cluster_rank() : 0;
  const int b = blockIdx.x / C;
  const int chunk = (V + C - 1) / C;
  const int lo = min(V, static_cast<int>(rank) * chunk), hi = min(V, lo + chunk);
  const int nrows = 2 * K + 1;                  // target rows 0..K, then draft rows 0..K-1
  auto row_ptr = [&](int r) -> const float* {
    return r <= K ? tl + (static_cast<int64_t>(b) * (K + 1) + r) * V
                  : dl + (static_cast<int64_t>(b) * K + (r - K - 1)) * V;
  };
  // ---- every row's statistics over this slice, then over the cluster --------------------------
  for (int r = 0; r < nrows; ++r) {
    float m, sm;
    slice_stats(row_ptr(r), lo, hi, sh, m, sm);
    if (threadIdx.x == 0) {
      part_m[r] = m;
      part_s[r] = sm;
    }
  }
  if (C > 1) cluster_sync();
  else __syncthreads();
  for (int r = threadIdx.x; r < nrows; r += kSpecThreads) {
    float M = -INFINITY;
    for (int c = 0; c < C; ++c) M = fmaxf(M, C > 1 ? ld_cluster_f32(part_m + r, c) : part_m[r]);
    float S = 0.f;
    for (int c = 0; c < C; ++c) {
      const float mc = C > 1 ? ld_cluster_f32(part_m + r, c) : part_m[r];
      const float sc = C > 1 ? ld_cluster_f32(part_s + r, c) : part_s[r];
      S += mc == -INFINITY ? 0.f : sc * exp_below(mc, M);
    }
    row_m[r] = M;
    row_s[r] = S;
  }
  __syncthreads();
  // ---- the accepted run (the same decisions in every CTA of the cluster) -----------------------
  int k = 0;
  for (; k < K; ++k) {
    const float* t = row_ptr(k);
    const float* d = row_ptr(K + 1 + k);
    const float mt = row_m[k], md = row_m[K + 1 + k];
    const float it = 1.f / row_s[k], id = 1.f / row_s[K + 1 + k];
    const int x = drafts[b * K + k];
    bool accept = false;
    if (x >= 0 && x < V) {
      const float pt = exp_below(t[x], mt) * it, pd = exp_below(d[x], md) * id;
      accept = ua[b * K + k] * pd < pt;
    } else if (threadIdx.x == 0 && rank == 0) {
      atomicOr(err, PKV_DEVERR_TOKEN);
    }
    if (accept) continue;
    const int nt = draw([&](int v) {
      return fmaxf(0.f, exp_below(__ldg(t + v), mt) * it - exp_below(__ldg(d + v), md) * id);
    }, lo, hi, V, us[b], sh, &slice_sum, &found, rank, C);
    if (threadIdx.x == 0 && nt >= 0) next_token[b] = nt;
    break;
  }
  if (k == K) {
    const float* t = row_ptr(K);
    const float mt = row_m[K], it = 1.f / row_s[K];
    const int nt = draw([&](int v) { return exp_below(__ldg(t + v), mt) * it; }, lo, hi, V,
                        us[b], sh, &slice_sum, &found, rank, C);
    if (threadIdx.x == 0 && nt >= 0) next_token[b] = nt;
  }
  if (threadIdx.x == 0 && rank == 0) n_accept[b] = k;
}

}  // namespace

extern "C" int pkv_spec_verify(const float* target_logits, const float* draft_logits,
                               const int32_t* drafts, const float* u_accept,
                               const float* u_sample, int num_seqs, int num_drafts, int vocab,
                               int32_t* n_accept, int32_t* next_token, pkv_stream_t stream) {
  if (num_seqs < 0 || num_drafts < 0 || vocab < 1 || 2 * num_drafts + 1 > kMaxRows)
    return PKV_EINVAL;
  if (num_seqs == 0) return PKV_OK;
  if (!target_logits || !u_sample || !n_accept || !next_token ||
      (num_drafts > 0 && (!draft_logits || !drafts || !u_accept)))
    return PKV_EINVAL;
  if (static_cast<int64_t>(num_seqs) * kMaxCluster >= (1ll << 31)) return PKV_EINVAL;
  unsigned int* err = pkv::device_error_ptr();
  if (!err) return pkv::cuda_status(cudaGetLastError());
  // CTAs per sequence: at least 2048 logits per CTA, up to a portable cluster of 8
  const int C = std::max(1, std::min(kMaxCluster, vocab / 2048));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(num_seqs * C));
  cfg.blockDim = dim3(kSpecThreads);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return pkv::cuda_status(cudaLaunchKernelEx(&cfg, spec_verify_kernel, target_logits,
                                             draft_logits, drafts, u_accept, u_sample,
                                             num_drafts, vocab, C, n_accept, next_token, err));
}
