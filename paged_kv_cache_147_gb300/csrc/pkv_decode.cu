// pkv_decode.cu -- paged decode attention and its sink + ring variant for sm_103a.
//
// What it computes ([VLLM] PagedAttention kernel paragraph; [EDGE] addressing section): each
// sequence's q_len newest query tokens, for each query head, attend over the sequence's cached
// K/V, which live in fixed-size physical blocks reached through the sequence's block table.
// The ring variant ([RING] §环形上下文与注意力沉淀机制) reads the sink + ring slots and rotates
// keys (RoPE) by their cache index at read time.
//
// Design (GB300):
//  * Work unit = (sequence b, kv head h). Every query head of the GQA group of h and every
//    query token of b forms one row of the unit's query tile (R = G * q_len rows), so each
//    K/V byte is read from HBM once for the whole group.
//  * The unit's context is cut into 16-token chunks (one chunk = 4 KB of K + 4 KB of V; a
//    block of bs tokens is bs/16 consecutive chunks). All units' chunks form one stream, in
//    which every unit is preceded by kSegCost empty positions (the cost of a segment in chunk
//    equivalents), and every CTA of a persistent grid (SM count x resident CTAs) takes an equal
//    contiguous slice of it: no CTA waits on a long sequence while others idle. A unit cut by
//    slice boundaries leaves normalised partials (m, l, o) in the workspace; the CTA holding
//    its first chunk merges them in slice order once the others have announced theirs (a
//    bounded wait; past it the last CTA to arrive merges instead, with the same partials in
//    the same order), so the result does not depend on scheduling or on which physical
//    blocks are used.
//  * One producer warp walks the slice, stages the block-table entries in registers (one
//    coalesced 32-entry load per 32 chunks: the block table never sits in the consumers'
//    path) and issues TMA tile loads (128-byte swizzle) of K and V into an NST-deep ring of
//    shared-memory stages, completing on mbarriers. The next chunks are in flight while the
//    consumers work on the current one.
//  * NCW consumer warps take the slice's chunks round-robin, each with its own online-softmax
//    state; an epilogue warp merges their states at each unit boundary and writes the output
//    or the partial. Scores and output come from mma.sync m16n8k16 (f16 in, f32 accumulate)
//    on ldmatrix fragments of the swizzled tiles: for up to 8 rows as S^T = K Q^T and
//    O^T = V^T P^T (keys and output dims on the mma's 16-row side), else as S = Q K^T and
//    O = P V with the rows padded to 16 or 32. Softmax runs in the exp2 domain; a row's
//    running maximum is refreshed (warp shuffles, rescale) only when a score exceeds it by
//    more than 2^8, so most steps take no warp-wide reduction.
//  * The fused-append launch may start while its predecessor finishes (programmatic
//    dependent launch): it requests its first stages, then waits for the predecessor before
//    touching queries, new K/V rows, outputs and the workspace.
//  * No wait is unbounded: an mbarrier wait gives up after kWaitLimit polls, sets
//    PKV_DEVERR_TIMEOUT and lets the kernel finish. Out-of-range block ids become
//    out-of-bounds TMA boxes (zero fill) and set PKV_DEVERR_BLOCK_ID.
#include <cuda_fp16.h>

#include <algorithm>
#include <atomic>
#include <map>
#include <mutex>
#include <tuple>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kD = 128;                       // head_dim
constexpr int kChunk = 16;                    // tokens per pipeline stage
constexpr int kHalfBytes = kChunk * 128;      // 16 rows x 64 dims x 2 B (one swizzled tile)
constexpr int kStageBytes = 4 * kHalfBytes;   // K lo/hi + V lo/hi = 8 KB
constexpr int kMaxCtasPerSm = 4;              // bounds the grid, hence the workspace
constexpr int kMaxSeqs = 4096;
// Per-segment cost in chunk equivalents: in the stream that is cut into equal slices, every
// non-empty unit is preceded by this many empty positions, so a CTA whose slice holds many
// short units (each one a segment: queries, hand-off, merge) gets fewer chunks.
#ifndef PKV_SEGMENT_COST
#define PKV_SEGMENT_COST 2
#endif
constexpr int kSegCost = PKV_SEGMENT_COST;
// Row stride (floats) of the per-warp output states in shared memory: 8 floats of padding put
// the 8 rows a warp's float2 stores touch at once in different banks.
constexpr int kSt = kD + 8;
constexpr float kNegInf = -__builtin_huge_valf();
// Consumer warps and pipeline stages per CTA, and the CTAs per SM the register budget of the
// one-m-tile kernels is sized for. Two consumer warps keep up with HBM (each takes a 16-token
// chunk in well under a microsecond) and leave the shared memory for ten 8 KB stages per CTA,
// two CTAs per SM: 160 KB of K/V in flight per SM.
#ifndef PKV_DECODE_WARPS
#define PKV_DECODE_WARPS 2
#endif
#ifndef PKV_DECODE_STAGES
#define PKV_DECODE_STAGES 10
#endif
#ifndef PKV_DECODE_MIN_CTAS
#define PKV_DECODE_MIN_CTAS 2
#endif
constexpr int kMinCtasMt1 = PKV_DECODE_MIN_CTAS;
// Ring kernels: resident CTAs per SM the register budget is sized for (the transposed-tile
// ones fit two CTAs per SM without spilling, the 16-row ones one).
#ifndef PKV_RING_MIN_CTAS
#define PKV_RING_MIN_CTAS 1
#endif
#ifndef PKV_RING_TR_MIN_CTAS
#define PKV_RING_TR_MIN_CTAS 2
#endif
// How long the CTA that merges a split unit waits for the unit's other partials before it
// falls back to announcing its own (normally they are in within microseconds).
#ifndef PKV_MERGE_WAIT_NS
#define PKV_MERGE_WAIT_NS 200000
#endif
constexpr uint64_t kMergeWaitNs = PKV_MERGE_WAIT_NS;

struct DecodeArgs {
  __half* out;
  const int32_t* block_tables;
  const int32_t* context_lens;  // paged
  const int64_t* logical_len;   // ring: L
  const int64_t* high_water;    // ring: hw
  const float* rope;            // ring: [sink + window][64][2] (cos, sin)
  float* part_o;                // [2 * grid][R][128]
  float* part_ml;               // [2 * grid][R][4]: m, l, 0, 0 (16-byte rows)
  int* counters;                // [num_seqs * Hkv]
  unsigned int* err;
  int num_blocks, max_blocks, num_seqs, q_len, Hq, Hkv, G, R;
  int block_size, bs_shift;     // bs_shift = log2(block_size / 16)
  int sink, window;
  float scale_log2;             // scale * log2(e)
  // fused append: this step's new K/V rows [B*q_len][Hkv][128] and the layer's pools
  const __half* k_new;
  const __half* v_new;
  __half* k_pool;
  __half* v_pool;
  // FP8 (E4M3) cache: per kv head scales of K and V (value = code * scale)
  const float* k_scale;
  const float* v_scale;
};

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------------------------------------
// Shared-memory layout (offsets from a 1024-byte aligned base).
template <int NCW, int NST, int MT, bool FP8 = false>
struct Smem {
  static constexpr int kNST = NST;
  // a stage holds one chunk's K and V (fp16, 8 KB) or two consecutive chunks' (E4M3, 8 KB: a
  // 32 x 128-byte K tile, then the V tile, whose codes the consumer warps widen in registers)
  static constexpr int kChunksPerStage = FP8 ? 2 : 1;
  static constexpr int kStage = FP8 ? 4 * kChunk * kD : kStageBytes;
  static constexpr int kQHalf = MT * 2048;            // 16*MT rows x 128 B
  static constexpr int kQBuf = 2 * kQHalf;
  static constexpr int kQ = NST * kStage;
  // full[NST], empty[NST], qfull[2], qempty[2], sdone[2], sfree[2]
  static constexpr int kBars = kQ + 2 * kQBuf;
  static constexpr int kFlags = kBars + (2 * NST + 8) * 8;  // abort, pending count + units
  static constexpr int kSrow = kFlags + 64;             // TMA row of each stage's chunks
  static constexpr int kState = kSrow + ((NST * 4 * kChunksPerStage + 15) & ~15);
  // segment states handed from the consumer warps to the epilogue warp, double-buffered:
  // o [2][NCW][R][kSt] (128 used), m [2][NCW][R], l [2][NCW][R]
  __host__ __device__ static int state_floats(int R) { return 2 * NCW * R * (kSt + 2); }
  __host__ __device__ static int seq_off(int R) { return kState + state_floats(R) * 4; }
  // per sequence: prefix (B+1 ints), length, high water; then (fused append) the new K/V
  // rows of the current segment, double-buffered with its queries: [2][q_len][K|V][256 B]
  __host__ __device__ static int newkv_off(int R, int B) {
    return (seq_off(R) + (3 * B + 1) * 4 + 127) & ~127;
  }
  __host__ static size_t bytes(int R, int B, int newkv_bytes) {
    return 1024 + static_cast<size_t>(newkv_off(R, B)) + static_cast<size_t>(newkv_bytes);
  }
};

struct Seg {
  int b, h, c0, c1, nb;  // chunks [c0, c1) of unit (b, h), which has nb chunks
  int x;                 // global stream index of chunk c0
};

// The stream: unit (b, h) of a sequence with nb > 0 chunks per kv head occupies nb + kSegCost
// positions, kSegCost empty ones and then its chunks; pre[b] is the length (per kv head) of the
// sequences before b, so the unit starts at pre[b] * Hkv + h * (nb + kSegCost). A CTA's slice
// [a, end) of the stream gives it segments: the runs of chunks of one unit inside the slice.
__device__ __forceinline__ int unit_first(const int* pre, int Hkv, int b, int h, int nb) {
  return pre[b] * Hkv + h * (nb + kSegCost) + kSegCost;   // position of the unit's chunk 0
}

struct Cursor {
  const int* pre;
  int B, Hkv, end;

  __device__ __forceinline__ bool first(int a, Seg& s) const {
    if (a >= end) return false;
    int lo = 0, hi = B - 1;  // largest b with pre[b] * Hkv <= a (a sequence with chunks)
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pre[mid] * Hkv <= a) lo = mid; else hi = mid - 1;
    }
    const int vl = pre[lo + 1] - pre[lo];
    const int off = a - pre[lo] * Hkv;
    const int h = off / vl, o = off - h * vl;
    const int ustart = a - o;
    const int x0 = ustart + kSegCost + max(o - kSegCost, 0);   // first chunk in the slice
    if (x0 >= end) return false;   // the slice ends before the unit's first chunk
    s.b = lo;
    s.h = h;
    s.nb = vl - kSegCost;
    s.c0 = x0 - ustart - kSegCost;
    s.c1 = min(s.nb, end - ustart - kSegCost);
    s.x = x0;
    return true;
  }
  __device__ __forceinline__ bool next(Seg& s) const {
    // the next unit's first chunk, if the slice reaches it (then this segment ended its unit)
    const int u2 = s.x - s.c0 + s.nb;
    if (u2 + kSegCost >= end) return false;
    if (++s.h == Hkv) {
      s.h = 0;
      do { ++s.b; } while (pre[s.b + 1] == pre[s.b]);
    }
    s.nb = pre[s.b + 1] - pre[s.b] - kSegCost;
    s.c0 = 0;
    s.c1 = min(s.nb, end - (u2 + kSegCost));
    s.x = u2 + kSegCost;
    return true;
  }
};

__device__ __forceinline__ void flag_timeout(const DecodeArgs& a, volatile int* abort) {
  atomicOr(a.err, PKV_DEVERR_TIMEOUT);
  *abort = 1;
}

// ---------------------------------------------------------------------------------------------
// Sync of the threads taking part in a merge: one warp, or a named barrier over NT threads.
template <int NT>
__device__ __forceinline__ void merge_sync() {
  if (NT == 32) __syncwarp();
  else named_barrier_sync(2, NT);
}

// Output row r (= query token qi, head g of the group) of unit (b, h): pointer to its 128 halves.
__device__ __forceinline__ __half* out_row(const DecodeArgs& a, int b, int h, int r) {
  const int qi = r / a.G, gg = r - qi * a.G;
  return a.out + ((static_cast<int64_t>(b) * a.q_len + qi) * a.Hq + h * a.G + gg) * kD;
}

__device__ __forceinline__ void store_half4(__half* dst, float4 v) {
  uint2 u;
  u.x = pack_half2(v.x, v.y);
  u.y = pack_half2(v.z, v.w);
  *reinterpret_cast<uint2*>(dst) = u;
}

// Weights of one row of a segment's per-warp states: w[ww] = 2^(m_ww - m) / l, with m the
// row's max and l = sum_ww l_ww 2^(m_ww - m); returns m and l for the partial.
template <int NCW>
__device__ __forceinline__ void row_weights(const float* m_s, const float* l_s, int R, int r,
                                            float (&w)[NCW], float& row_m, float& row_l) {
  row_m = kNegInf;
#pragma unroll
  for (int ww = 0; ww < NCW; ++ww) {
    w[ww] = m_s[ww * R + r];
    row_m = fmaxf(row_m, w[ww]);
  }
  row_l = 0.f;
#pragma unroll
  for (int ww = 0; ww < NCW; ++ww) {
    w[ww] = row_m == kNegInf ? 0.f : fast_exp2(w[ww] - row_m);
    row_l += l_s[ww * R + r] * w[ww];
  }
  const float inv = row_l > 0.f ? 1.f / row_l : 0.f;
#pragma unroll
  for (int ww = 0; ww < NCW; ++ww) w[ww] *= inv;
}

// Merge of one segment's per-warp states (o: [NCW][R] rows of kSt floats, unnormalised; m and
// l: [NCW][R]) into the unit's output (complete segment) or its normalised partial (split
// unit: rows of 128
// floats at po, rows of (m, l, 0, 0) at pml; global or shared memory), by NT threads
// t = 0..NT-1. Each thread owns 4 consecutive dims of a row (float4 in, 8 bytes out). One warp
// (NT == 32) forms each row's weights once, in lane r, and shares them by shuffle; a larger
// group has each thread form its own row's weights (the same arithmetic), with no barrier.
template <int NCW, int NT>
__device__ __forceinline__ void merge_segment(const DecodeArgs& a, const float* o_s,
                                              const float* m_s, const float* l_s, int b, int h,
                                              bool complete, float* po, float* pml, int t) {
  const int R = a.R;
  float w_own[NCW], m_own = 0.f, l_own = 0.f;
  if (NT == 32 && t < R) {
    row_weights<NCW>(m_s, l_s, R, t, w_own, m_own, l_own);
    if (!complete) *reinterpret_cast<float4*>(pml + t * 4) = make_float4(m_own, l_own, 0.f, 0.f);
  }
#pragma unroll 1
  for (int gi = t; gi < R * 32; gi += NT) {
    const int r = gi >> 5, c4 = gi & 31;
    float w[NCW];
    if (NT == 32) {
#pragma unroll
      for (int ww = 0; ww < NCW; ++ww) w[ww] = __shfl_sync(0xffffffffu, w_own[ww], r);
    } else {
      float row_m, row_l;
      row_weights<NCW>(m_s, l_s, R, r, w, row_m, row_l);
      if (!complete && c4 == 0)
        *reinterpret_cast<float4*>(pml + r * 4) = make_float4(row_m, row_l, 0.f, 0.f);
    }
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int ww = 0; ww < NCW; ++ww) {
      const float4 v = reinterpret_cast<const float4*>(o_s + (ww * R + r) * kSt)[c4];
      const float wt = w[ww];
      acc.x += wt * v.x; acc.y += wt * v.y; acc.z += wt * v.z; acc.w += wt * v.w;
    }
    if (complete)
      store_half4(out_row(a, b, h, r) + c4 * 4, acc);
    else
      reinterpret_cast<float4*>(po + r * kD)[c4] = acc;
  }
}

// The same merge of a segment's per-warp states by NT > 32 threads (the CTA's last segment, at
// the end of the launch): one thread per row forms the row's weights once and leaves them in
// the row's padding (floats kD.. of each state row), then every thread sums its own 4 dims.
template <int NCW, int NT>
__device__ __forceinline__ void merge_segment_wide(const DecodeArgs& a, float* o_s,
                                                   const float* m_s, const float* l_s, int b,
                                                   int h, bool complete, float* po, float* pml,
                                                   int t) {
  const int R = a.R;
  if (t < R) {
    float w[NCW], row_m, row_l;
    row_weights<NCW>(m_s, l_s, R, t, w, row_m, row_l);
#pragma unroll
    for (int ww = 0; ww < NCW; ++ww) o_s[(ww * R + t) * kSt + kD] = w[ww];
    if (!complete) *reinterpret_cast<float4*>(pml + t * 4) = make_float4(row_m, row_l, 0.f, 0.f);
  }
  named_barrier_sync(2, NT);
#pragma unroll 1
  for (int gi = t; gi < R * 32; gi += NT) {
    const int r = gi >> 5, c4 = gi & 31;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int ww = 0; ww < NCW; ++ww) {
      const float* row = o_s + (ww * R + r) * kSt;
      const float4 v = reinterpret_cast<const float4*>(row)[c4];
      const float wt = row[kD];
      acc.x += wt * v.x; acc.y += wt * v.y; acc.z += wt * v.z; acc.w += wt * v.w;
    }
    if (complete)
      store_half4(out_row(a, b, h, r) + c4 * 4, acc);
    else
      reinterpret_cast<float4*>(po + r * kD)[c4] = acc;
  }
}

// Where merge_unit stages partials in the (free) pipeline stage memory.
struct MergeStage {
  float* accv;    // [R][128] running output
  float* rowml;   // [2][R][2] running (max, sum), then [R][2] (scale of the running output,
                  // 1 / sum in the last batch) and [R][2] spare (keeps `so` 16-byte aligned)
  float* so;      // [PB][R][128] partials' o
  float* sml;     // [PB][R][4] partials' (m, l, weight, -)
  int PB;         // partials per batch (>= 2)
  __device__ MergeStage(uint8_t* stage_mem, int stage_bytes, int R) {
    accv = reinterpret_cast<float*>(stage_mem);
    rowml = accv + R * kD;
    PB = (stage_bytes - (R * kD + 8 * R) * 4) / (R * (kD + 4) * 4);
    so = rowml + 8 * R;
    sml = so + PB * R * kD;
  }
};

// Merge of a split unit's partials, run cooperatively by NT threads of the merging CTA (the one
// holding the unit's first chunk, or the last to arrive on the unit's counter), after its whole
// slice is done (so its pipeline stages are free).
// Partial p (in slice order) holds per row its max m_p, sum l_p and normalised output o_p; the
// result is sum_p o_p w_p / sum_p w_p with w_p = l_p 2^(m_p - M), M = max_p m_p, formed in slice
// order. The partials are copied into the stage memory with cp.async (as many per batch as fit,
// usually all: one round trip to L2); then one thread per row forms the row's weights, and every
// thread sums its own 4 output dims over the partials and divides by the row's sum. Each pass
// takes few dependent shared-memory round trips: this runs once per CTA at the end of the
// launch, where its latency is on the critical path.
// own >= 0: the unit's first partial (own == cf, the merging CTA's own) is already in the
// staging area, at index 0 of the first batch; it is not copied from the workspace.
template <int NT>
__device__ __forceinline__ void merge_unit(const DecodeArgs& a, int b, int h, int nb,
                                           const int* pre, int per, uint8_t* stage_mem,
                                           int stage_bytes, int t, int own = -1) {
  const int R = a.R;
  const int ua = unit_first(pre, a.Hkv, b, h, nb);
  const int cf = ua / per, cl = (ua + nb - 1) / per;
  // the unit is not the first segment of slice cf if that slice reaches back into the unit
  // before it (whose last chunk is the position just before this unit's empty ones)
  const bool first_odd = cf * per < ua - kSegCost;
  const MergeStage ms(stage_mem, stage_bytes, R);
  float* accv = ms.accv;
  float* rowml = ms.rowml;
  const int PB = ms.PB;
  float* so = ms.so;
  float* sml = ms.sml;   // per partial and row: m, l, then this batch's weight
  const uint32_t so_s = smem_u32(so), sml_s = smem_u32(sml);
  const int o_vec = R * kD / 4;                            // 16-byte pieces of one partial's o
  int batch = 0;
#pragma unroll 1
  for (int base = cf; base <= cl; base += PB, ++batch) {
    const int nbp = min(PB, cl - base + 1);
    const bool last_batch = base + PB > cl;
    merge_sync<NT>();                      // previous batch fully used
#pragma unroll 1
    for (int p = 0; p < nbp; ++p) {
      const int cc = base + p;
      if (cc == own) continue;
      const int64_t sl = 2 * cc + ((cc == cf && first_odd) ? 1 : 0);
      const float* src = a.part_o + sl * R * kD;
      const uint32_t dst = so_s + p * R * kD * 4;
      for (int i = t; i < o_vec; i += NT) cp_async_16(dst + i * 16, src + i * 4);
      if (t < R) cp_async_16(sml_s + (p * R + t) * 16, a.part_ml + (sl * R + t) * 4);
    }
    cp_async_wait_all();
    merge_sync<NT>();
    float* rsc = rowml + 4 * R;
    if (t < R) {
      // The row's (m, l) pairs are read into registers kRegP at a time (one shared-memory round
      // trip per group; a single one in the usual case of at most kRegP partials) before any
      // weight is written back.
      constexpr int kRegP = 8;
      const float* rin = rowml + (batch & 1) * 2 * R;
      float* rout = rowml + ((batch + 1) & 1) * 2 * R;
      const float M0 = batch ? rin[2 * t] : kNegInf;
      const float L0 = batch ? rin[2 * t + 1] : 0.f;
      float2 mlr[kRegP];
      float M = M0;
#pragma unroll 1
      for (int p0 = 0; p0 < nbp; p0 += kRegP) {
#pragma unroll
        for (int i = 0; i < kRegP; ++i) {
          const int p = p0 + i;
          mlr[i] = p < nbp ? *reinterpret_cast<const float2*>(sml + (p * R + t) * 4)
                           : make_float2(kNegInf, 0.f);
          M = fmaxf(M, mlr[i].x);
        }
      }
      const float sc = (M0 == kNegInf || M == kNegInf) ? 0.f : fast_exp2(M0 - M);
      float L = L0 * sc;
#pragma unroll 1
      for (int p0 = 0; p0 < nbp; p0 += kRegP) {
        if (nbp > kRegP) {
#pragma unroll
          for (int i = 0; i < kRegP; ++i) {
            const int p = p0 + i;
            mlr[i] = p < nbp ? *reinterpret_cast<const float2*>(sml + (p * R + t) * 4)
                             : make_float2(kNegInf, 0.f);
          }
        }
#pragma unroll
        for (int i = 0; i < kRegP; ++i) {
          const int p = p0 + i;
          const float wp = mlr[i].x == kNegInf ? 0.f : mlr[i].y * fast_exp2(mlr[i].x - M);
          L += wp;
          if (p < nbp) sml[(p * R + t) * 4 + 2] = wp;
        }
      }
      const float inv = !last_batch ? 1.f : (L > 0.f ? 1.f / L : 0.f);
      *reinterpret_cast<float2*>(rsc + 2 * t) = make_float2(sc, inv);
      rout[2 * t] = M;
      rout[2 * t + 1] = L;
    }
    merge_sync<NT>();
#pragma unroll 1
    for (int gi = t; gi < R * 32; gi += NT) {
      const int r = gi >> 5, c4 = gi & 31;
      const float2 si = *reinterpret_cast<const float2*>(rsc + 2 * r);
      float4 V = make_float4(0.f, 0.f, 0.f, 0.f);
      if (batch) {
        V = reinterpret_cast<const float4*>(accv)[gi];
        V.x *= si.x; V.y *= si.x; V.z *= si.x; V.w *= si.x;
      }
#pragma unroll 4
      for (int p = 0; p < nbp; ++p) {
        const float wp = sml[(p * R + r) * 4 + 2];
        const float4 o4 = reinterpret_cast<const float4*>(so + (p * R + r) * kD)[c4];
        V.x += wp * o4.x; V.y += wp * o4.y; V.z += wp * o4.z; V.w += wp * o4.w;
      }
      if (last_batch) {
        V.x *= si.y; V.y *= si.y; V.z *= si.y; V.w *= si.y;
        store_half4(out_row(a, b, h, r) + c4 * 4, V);
      } else {
        reinterpret_cast<float4*>(accv)[gi] = V;
      }
    }
  }
  if (t == 0) a.counters[b * a.Hkv + h] = 0;
  merge_sync<NT>();                        // stage memory free for the next merge
}

// Online softmax: a row's running maximum m is brought up to date (a warp-wide reduction and,
// if it grew, a rescale of l and O) only in a step where one of the row's scores exceeds m by
// more than this many powers of two. Any m with every score <= m + kLazyLog2 gives the same
// softmax: the weights exp2(x - m) stay <= 256, exact to fp16's relative precision, and the
// final 1 / l and the split merges use the same m as l and O.
constexpr float kLazyLog2 = 8.f;

// Word i (0-3) of a 16-byte vector (i a compile-time constant after unrolling).
__device__ __forceinline__ uint32_t u4_word(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Four E4M3 codes -> two fp16 pairs: bytes 0-1 into lo, bytes 2-3 into hi (exact).
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t x, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.rn.f16x2.e4m3x2 %0, l;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi) : "r"(x));
}

// Ring: rotate-half RoPE of one chunk's 16 keys by their cache index, in place in the chunk's K
// tile in shared memory (two 64-column halves at stK and stK + kHalfBytes, 128-byte swizzled),
// by one warp. Lane (p, q) = (lane % 8, lane / 8) takes the dim pairs (i, i + 64), i in
// [8 p, 8 p + 8), of keys 4 q .. 4 q + 3. Chunk c holds ring slots 16 c .. 16 c + 15; slot t's
// cache index is t for a sink, else sink + (t - r_lo) mod window. The factors cos / sin(j theta_i)
// of a group's first key come from the global table's row j; each next key whose index is one
// more is rotated on by the step factors cos / sin(theta_i) (the table's row 1, which stays in
// L1), a key after a jump in the index (the ring's wrap) reloads its row.
__device__ __forceinline__ void rope_pass(const DecodeArgs& a, uint32_t stK, int c, int r_lo,
                                          int lane) {
  const int cap = a.sink + a.window;
  const int p = lane & 7, q = lane >> 3;
  float step_c[8], step_s[8];
  {
    const float4* row = reinterpret_cast<const float4*>(a.rope) + (cap > 1 ? 32 : 0) + 4 * p;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float4 v = __ldg(row + u);
      step_c[2 * u] = v.x; step_s[2 * u] = v.y; step_c[2 * u + 1] = v.z; step_s[2 * u + 1] = v.w;
    }
  }
  float fc[8], fs[8];
  int jprev = -2;
#pragma unroll 1
  for (int kk = 0; kk < 4; ++kk) {
    const int r = 4 * q + kk;
    const int t = c * kChunk + r;
    int j = 0;
    if (t < a.sink) j = t;
    else if (t < cap) { int d = t - r_lo; if (d < 0) d += a.window; j = a.sink + d; }
    if (j != jprev + 1) {
      const float4* row = reinterpret_cast<const float4*>(a.rope) + j * 32 + 4 * p;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float4 v = __ldg(row + u);
        fc[2 * u] = v.x; fs[2 * u] = v.y; fc[2 * u + 1] = v.z; fs[2 * u + 1] = v.w;
      }
    } else {
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float c2 = fc[u] * step_c[u] - fs[u] * step_s[u];
        fs[u] = fs[u] * step_c[u] + fc[u] * step_s[u];
        fc[u] = c2;
      }
    }
    jprev = j;
    const uint32_t px = stK + swz128(r, p);                // dims 8 p .. 8 p + 7
    const uint32_t py = stK + kHalfBytes + swz128(r, p);   // dims 64 + 8 p ..
    const uint4 xv = ld_shared_v4(px), yv = ld_shared_v4(py);
    const uint32_t xs[4] = {xv.x, xv.y, xv.z, xv.w}, ys[4] = {yv.x, yv.y, yv.z, yv.w};
    uint32_t xo[4], yo[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float2 x = __half22float2(*reinterpret_cast<const __half2*>(&xs[u]));
      const float2 y = __half22float2(*reinterpret_cast<const __half2*>(&ys[u]));
      const float c0 = fc[2 * u], s0 = fs[2 * u], c1 = fc[2 * u + 1], s1 = fs[2 * u + 1];
      xo[u] = pack_half2(x.x * c0 - y.x * s0, x.y * c1 - y.y * s1);
      yo[u] = pack_half2(y.x * c0 + x.x * s0, y.y * c1 + x.y * s1);
    }
    st_shared_v4(px, make_uint4(xo[0], xo[1], xo[2], xo[3]));
    st_shared_v4(py, make_uint4(yo[0], yo[1], yo[2], yo[3]));
  }
}

// Ring: starts the factor rows rope_pass will load for chunk c (the first key of each lane's
// 4-key group) towards L1, one chunk ahead of their use (lane (p, q): 64 bytes of row j(16 c +
// 4 q), the part of the row its dims need).
__device__ __forceinline__ void rope_prefetch(const DecodeArgs& a, int c, int r_lo, int lane) {
  const int cap = a.sink + a.window;
  const int t = c * kChunk + 4 * (lane >> 3);
  int j = 0;
  if (t < a.sink) j = t;
  else if (t < cap) { int d = t - r_lo; if (d < 0) d += a.window; j = a.sink + d; }
  prefetch_l1(a.rope + j * 128 + 16 * (lane & 7));
}

// Ring: logical position held by ring slot t of a sequence whose window part starts at position
// lo_pos (in slot r_lo), or INT_MAX for a slot past the ring's capacity.
__device__ __forceinline__ int ring_pos(const DecodeArgs& a, int t, int lo_pos, int r_lo) {
  if (t < a.sink) return t;
  if (t >= a.sink + a.window) return 0x7fffffff;
  int d = t - r_lo;
  if (d < 0) d += a.window;
  return lo_pos + d;
}

// Requests segment kk's queries (and, fused append, its new K/V rows) into query buffer kk & 1,
// completing on that buffer's full barrier; waits first until the consumers have released the
// buffer's previous use. One thread.
template <class L, bool APPEND>
__device__ __forceinline__ void issue_queries(const DecodeArgs& a, const CUtensorMap* tmQ,
                                              uint32_t sbase, int B, const Seg& sg, int kk,
                                              volatile int* abort) {
  const uint32_t bar_qfull = sbase + L::kBars + 2 * L::kNST * 8;
  const uint32_t bar_qempty = bar_qfull + 2 * 8;
  const int qs = kk & 1;
  if (kk >= 2 && !mbar_wait(bar_qempty + qs * 8, ((kk >> 1) - 1) & 1, abort))
    flag_timeout(a, abort);
  mbar_arrive_expect_tx(bar_qfull + qs * 8, a.R * 256 + (APPEND ? a.q_len * 512 : 0));
  const uint32_t qdst = sbase + L::kQ + qs * L::kQBuf;
  tma_load_3d(qdst, tmQ, 0, sg.h * a.G, sg.b * a.q_len, bar_qfull + qs * 8);
  tma_load_3d(qdst + L::kQHalf, tmQ, 64, sg.h * a.G, sg.b * a.q_len, bar_qfull + qs * 8);
  if (APPEND) {
    const uint32_t nkv = sbase + L::newkv_off(a.R, B) + qs * a.q_len * 512;
    for (int i = 0; i < a.q_len; ++i) {
      const int64_t row = (static_cast<int64_t>(sg.b) * a.q_len + i) * a.Hkv + sg.h;
      bulk_load(nkv + i * 512, a.k_new + row * kD, 256, bar_qfull + qs * 8);
      bulk_load(nkv + i * 512 + 256, a.v_new + row * kD, 256, bar_qfull + qs * 8);
    }
  }
}

// ---------------------------------------------------------------------------------------------
// Warp roles: warps 0..NCW-1 consume chunks, warp NCW produces (TMA), warp NCW+1 is the
// epilogue (merges each segment's per-warp states, writes outputs and split-unit partials,
// announces arrivals), so the consumers never stop at a unit boundary.
template <int NCW, int NST, int MT, bool RING, bool APPEND, bool TR, bool FP8, bool KV3D>
__global__ void __launch_bounds__((NCW + 2) * 32,
                                  MT != 1 ? 1
                                  : RING  ? (TR ? PKV_RING_TR_MIN_CTAS : PKV_RING_MIN_CTAS)
                                          : kMinCtasMt1)
decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
              const __grid_constant__ CUtensorMap tmQ, const DecodeArgs a) {
  using L = Smem<NCW, NST, MT, FP8>;
  // Stage st holds the CTA's chunks st, st + NST, ... and chunk j goes to consumer warp
  // j % NCW. With NST a multiple of NCW every use of a stage goes to the same warp, which
  // takes them in order, so it never waits on a full-barrier phase more than one ahead of the
  // last completed one (all that a parity wait can tell apart).
  static_assert(NST % NCW == 0, "pipeline stages must be a multiple of the consumer warps");
  static_assert(!TR || MT == 1, "the transposed tile is for up to 8 rows");
  static_assert(!(FP8 && RING), "the E4M3 cache is paged only");
  static_assert(!FP8 || TR, "the E4M3 cache is read by the transposed tile only");
  static_assert(!KV3D || !FP8, "the 3-D K/V boxes are for the fp16 cache");
  // the queries' buffer stays in use for the whole segment when its fragments are not kept in
  // registers, or when it also holds the segment's new K/V rows
  constexpr bool kHoldQ = MT != 1 || APPEND;
  constexpr int kNC = NCW * 32;          // consumer threads
  constexpr int kNE = (NCW + 1) * 32;    // consumers + epilogue (final merges)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + L::kBars;
  const uint32_t bar_empty = bar_full + NST * 8;
  const uint32_t bar_qfull = bar_empty + NST * 8;
  const uint32_t bar_qempty = bar_qfull + 2 * 8;
  const uint32_t bar_sdone = bar_qempty + 2 * 8;
  const uint32_t bar_sfree = bar_sdone + 2 * 8;
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::kFlags);
  int* srow_s = reinterpret_cast<int*>(smem + L::kSrow);
  int* npend_s = reinterpret_cast<int*>(smem + L::kFlags) + 1;   // then 2 x (b, h, nb)
  volatile int* fast_s = reinterpret_cast<volatile int*>(smem + L::kFlags) + 8;
  float* stO = reinterpret_cast<float*>(smem + L::kState);     // [2][NCW][R][kSt]
  float* stM = stO + 2 * NCW * a.R * kSt;                       // [2][NCW][R]
  float* stL = stM + 2 * NCW * a.R;                             // [2][NCW][R]
  int* pre = reinterpret_cast<int*>(smem + L::seq_off(a.R));
  int* slen = pre + a.num_seqs + 1;   // ctx (paged) or L (ring), clamped
  int* shw = slen + a.num_seqs;       // ring: high water

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int B = a.num_seqs;
  const int cap = a.sink + a.window;

  // ---- per-sequence lengths and chunk counts -------------------------------------------------
  for (int b = tid; b < B; b += blockDim.x) {
    int len, nchunks, hw = 0;
    if (!RING) {
      int ctx = a.context_lens[b];
      const int lim = a.max_blocks * a.block_size;
      if (ctx < 0 || ctx > lim) {
        atomicOr(a.err, PKV_DEVERR_CONTEXT);
        ctx = ctx < 0 ? 0 : lim;
      }
      len = ctx;
      nchunks = (ctx + kChunk - 1) / kChunk;
    } else {
      long long Lb = a.logical_len[b], hb = a.high_water[b];
      if (Lb < 0 || Lb > 0x3fffffffLL) { atomicOr(a.err, PKV_DEVERR_CONTEXT); Lb = Lb < 0 ? 0 : 0x3fffffff; }
      if (hb < Lb) hb = Lb;
      if (hb > 0x3fffffffLL) hb = 0x3fffffff;
      len = static_cast<int>(Lb);
      hw = static_cast<int>(hb);
      nchunks = (min(hw, cap) + kChunk - 1) / kChunk;
    }
    slen[b] = len;
    shw[b] = hw;
    pre[b + 1] = nchunks > 0 ? nchunks + kSegCost : 0;  // scanned below
  }
  // zero both Q buffers so rows past R are finite; TMA overwrites rows < R
  for (int i = tid; i < L::kQBuf * 2 / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(smem + L::kQ)[i] = make_uint4(0, 0, 0, 0);
  if (tid == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(bar_full + s * 8, 1);
      mbar_init(bar_empty + s * 8, 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar_qfull + s * 8, 1);
      mbar_init(bar_qempty + s * 8, NCW);
      mbar_init(bar_sdone + s * 8, NCW);
      mbar_init(bar_sfree + s * 8, 1);
    }
    *abort = 0;
    *npend_s = 0;
    pre[0] = 0;
  }
  fence_barrier_init();
  __syncthreads();
  // inclusive scan of chunk counts (warp 0: contiguous slices per lane + shuffle scan)
  if (warp == 0) {
    const int per_lane = (B + 31) / 32;
    const int lo = min(B, lane * per_lane), hi = min(B, lo + per_lane);
    int sum = 0;
    for (int b = lo; b < hi; ++b) sum += pre[b + 1];
    int incl = sum;
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - sum;
    for (int b = lo; b < hi; ++b) {
      run += pre[b + 1];
      pre[b + 1] = run;
    }
  }
  __syncthreads();

  const int total = pre[B] * a.Hkv;
  const int per = (total + gridDim.x - 1) / gridDim.x;
  const int begin = blockIdx.x * per;
  const Cursor cur{pre, B, a.Hkv, min(total, begin + per)};

  // let the next kernel on the stream launch as soon as SM resources free up (its own
  // dependency wait keeps it from reading anything this kernel writes)
  if (tid == 0) griddep_launch_dependents();

  if (warp == NCW) {
    // =================================== producer ============================================
    const int chunk_mask = (1 << a.bs_shift) - 1;
    const uint64_t kv_policy = l2_policy_evict_first();
    int j = 0, k = 0;
    Seg s;
    bool has = cur.first(begin, s);
    // block-table entries of the next 32 chunks, loaded one group ahead of their use
    auto load_ids = [&](const Seg& sg, int cb) -> int32_t {
      const int cc = cb + lane;
      return cc < sg.c1 ? __ldg(a.block_tables + static_cast<int64_t>(sg.b) * a.max_blocks +
                                (cc >> a.bs_shift))
                        : -1;
    };
    int32_t ids = has ? load_ids(s, s.c0) : -1;
    if (lane == 0) {
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
      prefetch_tensormap(&tmQ);
    }
    // The fused-append variant may be launched before the preceding kernel on the stream has
    // finished (programmatic dependent launch). Its K/V pool, block tables and context lengths
    // are not written by that kernel, so the first NST chunks are requested right away; the
    // queries, the new K/V rows, the output and the workspace are touched only after
    // griddepcontrol.wait. The other variants wait before their first query load (a no-op,
    // as they are never launched early).
    const bool early_kv = APPEND;
    bool waited = false;
    auto issue_q = [&](const Seg& sg, int kk) {
      if (lane == 0) issue_queries<L, APPEND>(a, &tmQ, sbase, B, sg, kk, abort);
    };
    while (has) {
      // with an early start the epilogue warp requests the first segment's queries (it is
      // idle until a segment ends): they go out as soon as the dependency is met, while
      // this warp is still filling the stages
      if (!early_kv || k > 0) {
        if (!waited) { griddep_wait(); waited = true; }
        issue_q(s, k);
      }
      Seg nx = s;
      const bool has_next = cur.next(nx);
      for (int cb = s.c0; cb < s.c1; cb += 32) {
        const int32_t cur_ids = ids;
        // prefetch the next group: the rest of this segment, or the next segment's start
        if (cb + 32 < s.c1) ids = load_ids(s, cb + 32);
        else if (has_next) ids = load_ids(nx, nx.c0);
        const int cc = cb + lane;
        int row = -kChunk;  // an out-of-range box: TMA fills it with zeros
        if (cc < s.c1) {
          if (cur_ids >= 0 && cur_ids < a.num_blocks)
            row = (cur_ids * a.Hkv + s.h) * a.block_size + ((cc & chunk_mask) << 4);
          else
            atomicOr(a.err, PKV_DEVERR_BLOCK_ID);
        }
        const int n = min(32, s.c1 - cb);
        // E4M3: a stage takes chunks l and l + 1 of this group (l + 1 past the segment's end is
        // an out-of-range row: an all-zero box)
        for (int l = 0; l < n; l += L::kChunksPerStage, ++j) {
          if (early_kv && !waited && j == NST) {
            // every stage is requested; none frees before the dependency is met
            griddep_wait();
            waited = true;
          }
          const int r = __shfl_sync(0xffffffffu, row, l);
          const int r2 = FP8 ? __shfl_sync(0xffffffffu, row, (l + 1) & 31) : 0;
          const int st = j % NST;
          const uint32_t fb = bar_full + st * 8;
          if (lane == 0) {
            if (j >= NST && !mbar_wait(bar_empty + st * 8, ((j / NST) - 1) & 1, abort))
              flag_timeout(a, abort);
            // published to the consumer by the barrier below
            if (APPEND) {
              srow_s[L::kChunksPerStage * st] = r;
              if (FP8) srow_s[2 * st + 1] = r2;
            }
            mbar_arrive_expect_tx(fb, L::kStage);
          }
          __syncwarp();                   // the stage is free before any lane writes it
          // The chunk's boxes go out as one warp instruction from several lanes: a tensor copy
          // costs its issuing thread tens of cycles, and one thread issuing all of a chunk's
          // copies held each chunk up ~150 ns. K/V are read once per step: first to go from
          // L2, which then keeps the partials, queries and tables the merges and other CTAs
          // need.
          if (FP8) {
            // E4M3: 2 KB boxes (16 rows x 128 bytes): K of both chunks, then V of both
            if (lane < 4)
              tma_load_2d_hint(sbase + st * L::kStage + lane * (kChunk * kD),
                               (lane >> 1) ? &tmV : &tmK, 0, (lane & 1) ? r2 : r, fb, kv_policy);
          } else if (KV3D) {
            // one box each for K (lane 0) and V (lane 1), both 64-column halves of the chunk's
            // 16 rows (4 KB, two 128-byte-swizzled 2 KB tiles)
            if (lane < 2)
              tma_load_3d_hint(sbase + st * kStageBytes + lane * 2 * kHalfBytes,
                               lane ? &tmV : &tmK, 0, r, 0, fb, kv_policy);
          } else if (lane < 4) {
            // one box each for the 64-column halves of K (lanes 0, 1) and V (lanes 2, 3)
            tma_load_2d_hint(sbase + st * kStageBytes + lane * kHalfBytes, lane < 2 ? &tmK : &tmV,
                             (lane & 1) * 64, r, fb, kv_policy);
          }
        }
      }
      ++k;
      s = nx;
      has = has_next;
    }
    if (!waited) griddep_wait();
    // sequences without any chunk get zeros (their units are in no CTA's slice)
    for (int b = blockIdx.x; b < B; b += gridDim.x) {
      if (pre[b + 1] != pre[b]) continue;
      const int n = a.q_len * a.Hq * kD;
      for (int i = lane; i < n; i += 32)
        a.out[static_cast<int64_t>(b) * n + i] = __float2half_rn(0.f);
    }
    // Before exiting, make sure no TMA write into this CTA's shared memory is still pending
    // (only matters if the consumers gave up early; otherwise these waits return at once).
    if (lane == 0) {
      for (int jj = max(0, j - NST); jj < j; ++jj)
        if (!mbar_wait(bar_full + (jj % NST) * 8, (jj / NST) & 1, nullptr)) flag_timeout(a, abort);
      for (int kk = max(0, k - 2); kk < k; ++kk)
        if (!mbar_wait(bar_qfull + (kk & 1) * 8, (kk >> 1) & 1, nullptr)) flag_timeout(a, abort);
    }
    return;
  }

  // the CTA's last segment (merged at the end by consumers and epilogue together)
  int last_k = -1, last_b = 0, last_h = 0, last_nb = 0, last_slot = 0;
  bool last_complete = true, last_head = false;
  {
    Seg s;
    bool has = cur.first(begin, s);
    int kk = 0;
    while (has) {
      last_k = kk;
      last_b = s.b; last_h = s.h; last_nb = s.nb;
      last_complete = (s.c0 == 0 && s.c1 == s.nb);
      last_head = s.c0 == 0;
      last_slot = 2 * blockIdx.x + (kk == 0 ? 0 : 1);
      ++kk;
      has = cur.next(s);
    }
  }

  if (warp == NCW + 1) {
    // =================================== epilogue ============================================
    // Merges every segment but the last as soon as the consumers hand it over, writes the
    // output (or the partial of a split unit) and announces split units' arrivals.
    int k = 0, npend = 0;
    Seg s;
    bool has = cur.first(begin, s);
    if (APPEND && has) {
      griddep_wait();
      if (lane == 0) issue_queries<L, APPEND>(a, &tmQ, sbase, B, s, 0, abort);
    }
    while (has && k < last_k) {
      const int sb = k & 1;
      if (!mbar_wait(bar_sdone + sb * 8, (k >> 1) & 1, abort)) flag_timeout(a, abort);
      const bool complete = (s.c0 == 0 && s.c1 == s.nb);
      const int slot = 2 * blockIdx.x + (k == 0 ? 0 : 1);
      merge_segment<NCW, 32>(a, stO + sb * NCW * a.R * kSt, stM + sb * NCW * a.R,
                             stL + sb * NCW * a.R, s.b, s.h, complete,
                             a.part_o + static_cast<int64_t>(slot) * a.R * kD,
                             a.part_ml + static_cast<int64_t>(slot) * a.R * 4, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_sfree + sb * 8);
      if (!complete) {
        // Announce the partial. The warp barrier orders the other lanes' writes before lane
        // 0's arrival, a gpu-scope acquire-release atomic: the release publishes the partial,
        // and a last arrival's acquire makes the other CTAs' partials visible. That merge waits
        // for the end of the slice, when the whole CTA can do it.
        if (lane == 0) {
          const int ua = unit_first(pre, a.Hkv, s.b, s.h, s.nb);
          const int parts = (ua + s.nb - 1) / per - ua / per + 1;
          if (atomic_add_acq_rel(a.counters + s.b * a.Hkv + s.h, 1) == parts - 1) {
            npend_s[1 + 3 * npend] = s.b;
            npend_s[2 + 3 * npend] = s.h;
            npend_s[3 + 3 * npend] = s.nb;
            ++npend;
          }
        }
      }
      ++k;
      has = cur.next(s);
    }
    if (lane == 0) *npend_s = npend;
  } else {
    // =================================== consumers ===========================================
    const int w = warp;
    const int g = lane >> 2, t4 = lane & 3;
    int j = 0, k = 0;
    Seg s;
    bool has = cur.first(begin, s);
    while (has) {
      const int qs = k & 1;
      const uint32_t qb = sbase + L::kQ + qs * L::kQBuf;
      if (!mbar_wait(bar_qfull + qs * 8, (k >> 1) & 1, abort)) flag_timeout(a, abort);

      const int Lc = slen[s.b];  // tokens in cache (paged ctx / ring L)
      int lo_pos = 0, r_lo = 0;
      if (RING) {
        const int hw = shw[s.b];
        lo_pos = max(a.sink, hw - a.window);
        r_lo = a.sink + (lo_pos - a.sink) % a.window;
        // rotate this segment's query rows in place by their own cache index
        for (int idx = tid; idx < a.R * 64; idx += kNC) {
          const int r = idx >> 6, d = idx & 63;
          const int pos = Lc - a.q_len + r / a.G;
          int jq = pos < a.sink ? pos : a.sink + (pos - lo_pos);
          jq = min(max(jq, 0), cap - 1);
          const uint32_t off = swz128(r, d >> 3) + (d & 7) * 2;
          __half* px = reinterpret_cast<__half*>(smem + (qb - sbase) + off);
          __half* py = reinterpret_cast<__half*>(smem + (qb - sbase) + L::kQHalf + off);
          const float2 cs = __ldg(reinterpret_cast<const float2*>(a.rope) + jq * 64 + d);
          const float x = __half2float(*px), y = __half2float(*py);
          *px = __float2half_rn(x * cs.x - y * cs.y);
          *py = __float2half_rn(y * cs.x + x * cs.y);
        }
        named_barrier_sync(1, kNC);   // consumers only
      }

      if constexpr (TR) {
      // ---- up to 8 rows: the transposed tile. S^T = K Q^T and O^T = V^T P^T, so the 16 keys
      // of a chunk (and 16 dims of O) fill the mma's 16-row side and the (at most 8) query rows
      // its 8 columns: half the mma of the 16-row form, half the accumulators. Thread (g, t4)
      // holds rows 2t4 and 2t4 + 1 of the group, keys g and g + 8, dims 16 dt + g (+ 8).
      // Q^T fragments (B operand): rows 0-7 of the query tile
      uint32_t qb0[8], qb1[8];
      if constexpr (FP8) {
        // E4M3 keys: thread t4 takes dims 16 s8 + 4 t4 .. + 3 of every 16-dim step as its
        // fragment columns 2 t4, 2 t4 + 1, 2 t4 + 8, 2 t4 + 9 (a reordering of the summed
        // dimension, the same for keys and queries), so that its four key codes are one
        // 32-bit word of a row
#pragma unroll
        for (int s8 = 0; s8 < 8; ++s8) {
          const int d0 = 16 * s8 + 4 * t4;
          const uint2 qq = ld_shared_v2(qb + (d0 >> 6) * L::kQHalf + swz128(g, (d0 & 63) >> 3) +
                                        (d0 & 7) * 2);
          qb0[s8] = qq.x;
          qb1[s8] = qq.y;
        }
      } else {
#pragma unroll
        for (int s8 = 0; s8 < 8; ++s8) {
          const int i = lane >> 3;
          const int row = (i & 1) * 8 + (lane & 7);
          const int ch = 2 * s8 + (i >> 1);
          uint32_t unused0, unused1;
          ldsm_x4(qb + (ch >> 3) * L::kQHalf + swz128(row, ch & 7), qb0[s8], unused0, qb1[s8],
                  unused1);
        }
      }
      if (!kHoldQ) {
        if (RING) fence_proxy_async_smem();   // the queries were rotated in place
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_qempty + qs * 8);
      }
      float tm[2] = {kNegInf, kNegInf}, tl[2] = {0.f, 0.f}, ot[8][4];
#pragma unroll
      for (int dt = 0; dt < 8; ++dt) ot[dt][0] = ot[dt][1] = ot[dt][2] = ot[dt][3] = 0.f;
      int tlim[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int r = 2 * t4 + e;
        const int qi = r < a.R ? r / a.G : a.q_len - 1;
        tlim[e] = Lc - a.q_len + qi + 1;
      }
      // E4M3 cache: the kv head's K scale joins the score scale, its V scale the output
      const float score_l2 = FP8 ? a.scale_log2 * __ldg(a.k_scale + s.h) : a.scale_log2;
      const float out_sc = FP8 ? __ldg(a.v_scale + s.h) : 1.f;
      const int nchunk = s.c1 - s.c0;
      if constexpr (FP8) {
        // ---- E4M3: a stage holds chunks c and c + 1 of the segment (c + 1 an all-zero box
        // past its end when the segment has an odd number of chunks). A warp takes whole
        // stages: 32 keys per online-softmax step, two independent mma chains per product.
        const int npair = (nchunk + 1) >> 1;
        for (int jp = ((w - j) % NCW + NCW) % NCW; jp < npair; jp += NCW) {
          const int gj = j + jp;
          const int st = gj % NST;
          if (!mbar_wait(bar_full + st * 8, (gj / NST) & 1, abort)) flag_timeout(a, abort);
          const uint32_t stK = sbase + st * L::kStage;   // rows 0-15: chunk c, 16-31: c + 1
          const uint32_t stVc = stK + 2 * kChunk * kD;
          const int c = s.c0 + 2 * jp;
          const bool two = c + 1 < s.c1;
          const int nk = two ? 2 * kChunk : kChunk;      // keys of the segment in the stage
          const bool full = two && (c + 2) * kChunk <= Lc - a.q_len + 1;
          bool patched = false;
          if (APPEND && (c * kChunk + nk > Lc - a.q_len)) {
            // lanes 0-7 quantise a 16-element piece of a new K row, 8-15 of the V row (divided
            // by the head's scale in binary32, as pkv_kv_append_fp8 does), into the stage's
            // code tiles and the pool
            const int first_new = Lc - a.q_len;
            const uint32_t nkv = sbase + L::newkv_off(a.R, B) + qs * a.q_len * 512;
            const int which = (lane >> 3) & 1, p = lane & 7;
            const float sc = __ldg((which ? a.v_scale : a.k_scale) + s.h);
            for (int i = 0; i < a.q_len; ++i) {
              const int pos = first_new + i;
              const int tk = pos - c * kChunk;   // row in the stage's 32-row tiles
              if (lane >= 16 || pos < 0 || tk < 0 || tk >= nk) continue;
              const uint4 h0 = ld_shared_v4(nkv + i * 512 + which * 256 + p * 32);
              const uint4 h1 = ld_shared_v4(nkv + i * 512 + which * 256 + p * 32 + 16);
              const uint4 q8 = make_uint4(f16x4_to_e4m3x4(h0.x, h0.y, sc),
                                          f16x4_to_e4m3x4(h0.z, h0.w, sc),
                                          f16x4_to_e4m3x4(h1.x, h1.y, sc),
                                          f16x4_to_e4m3x4(h1.z, h1.w, sc));
              st_shared_v4(stK + which * (2 * kChunk * kD) + swz128(tk, p), q8);
              const int srow = srow_s[2 * st + (tk >> 4)];
              if (srow >= 0) {
                uint8_t* pool = reinterpret_cast<uint8_t*>(which ? a.v_pool : a.k_pool);
                *reinterpret_cast<uint4*>(pool + (static_cast<int64_t>(srow) + (tk & 15)) * kD +
                                          p * 16) = q8;
              }
            }
            __syncwarp();
            patched = true;
          }
          // ---- the stage's codes into registers, then the stage goes back to the producer:
          // K, keys g and g + 8 of each chunk, one word of four codes per 16-dim step; V, dims
          // 16 g .. 16 g + 15 of keys 2 t4, 2 t4 + 1, 2 t4 + 8, 2 t4 + 9 of each chunk (the
          // output dims of rows g and g + 8 of the PV tiles below) ----
          uint32_t kw[2][8][2];
          uint4 vr[2][4];
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              kw[h][ks][0] = ld_shared_u32(stK + swz128(16 * h + g, ks) + 4 * t4);
              kw[h][ks][1] = ld_shared_u32(stK + swz128(16 * h + g + 8, ks) + 4 * t4);
            }
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int i = 0; i < 4; ++i)
              vr[h][i] = ld_shared_v4(stVc + swz128(16 * h + 2 * t4 + (i & 1) + 8 * (i >> 1), g));
          if (APPEND && patched) fence_proxy_async_smem();
          __syncwarp();                      // every code of the stage has been read
          if (lane == 0) mbar_arrive(bar_empty + st * 8);
          // ---- S^T = K Q^T for both chunks, the codes widened in registers; two chains per
          // chunk ----
          float sa[2][4], sb[2][4];
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int i = 0; i < 4; ++i) sa[h][i] = sb[h][i] = 0.f;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              uint32_t a0, a1, a2, a3;
              e4m3x4_to_f16x4(kw[h][ks][0], a0, a2);
              e4m3x4_to_f16x4(kw[h][ks][1], a1, a3);
              if (ks & 1)
                mma_16816(sb[h], a0, a1, a2, a3, qb0[ks], qb1[ks]);
              else
                mma_16816(sa[h], a0, a1, a2, a3, qb0[ks], qb1[ks]);
            }
          }

          // ---- mask, online softmax over this thread's rows and 4 keys (exp2 domain). The
          // running maximum is only brought up to date when a score exceeds it by more than
          // kLazyLog2 (so every weight stays <= 2^kLazyLog2, exact in fp16 and fp32 alike); else
          // the step needs no warp-wide reduction and no rescale ----
          float pv[2][4], alpha[2] = {1.f, 1.f};
          float x[2][2][2];   // [row e][chunk h][key g, g + 8]
          bool grow = false;
#pragma unroll
          for (int e = 0; e < 2; ++e) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              x[e][h][0] = (sa[h][e] + sb[h][e]) * score_l2;           // key g of chunk c + h
              x[e][h][1] = (sa[h][2 + e] + sb[h][2 + e]) * score_l2;   // key g + 8
              if (!full) {
                const int p0 = (c + h) * kChunk + g;
                const bool ok = h == 0 || two;
                x[e][h][0] = ok && p0 < tlim[e] ? x[e][h][0] : kNegInf;
                x[e][h][1] = ok && p0 + 8 < tlim[e] ? x[e][h][1] : kNegInf;
              }
            }
            const float lm = fmaxf(fmaxf(x[e][0][0], x[e][0][1]), fmaxf(x[e][1][0], x[e][1][1]));
            grow |= lm > tm[e] + kLazyLog2;
          }
          if (__any_sync(0xffffffffu, grow)) {
            bool rescale = false;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              float mx = fmaxf(fmaxf(x[e][0][0], x[e][0][1]), fmaxf(x[e][1][0], x[e][1][1]));
              mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
              mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
              mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
              const float m_old = tm[e];
              const float m_new = fmaxf(m_old, mx);
              const float m_use = m_new == kNegInf ? 0.f : m_new;
              alpha[e] = fast_exp2(m_old - m_use);
              rescale |= (m_old != kNegInf) && (m_new != m_old);
              tm[e] = m_new;
            }
            if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
              for (int dt = 0; dt < 8; ++dt) {
                ot[dt][0] *= alpha[0];
                ot[dt][1] *= alpha[1];
                ot[dt][2] *= alpha[0];
                ot[dt][3] *= alpha[1];
              }
            }
          }
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float m_use = tm[e] == kNegInf ? 0.f : tm[e];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              pv[h][e] = fast_exp2(x[e][h][0] - m_use);
              pv[h][2 + e] = fast_exp2(x[e][h][1] - m_use);
            }
            tl[e] = tl[e] * alpha[e] + ((pv[0][e] + pv[0][2 + e]) + (pv[1][e] + pv[1][2 + e]));
          }
          // P^T of each chunk (keys x rows) to the B operand: transpose the two 8x8 halves
          uint32_t pb[2][2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            pb[h][0] = movmatrix_trans(pack_half2(pv[h][0], pv[h][1]));
            pb[h][1] = movmatrix_trans(pack_half2(pv[h][2], pv[h][3]));
          }
          // tokens no query may see may hold anything, NaN included: zero their V entries
          uint32_t vm[2][2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            vm[h][0] = vm[h][1] = 0xffffffffu;
            if (!full) {
              const int t0 = (c + h) * kChunk + 2 * t4;
              const int lim = (h == 0 || two) ? Lc : 0;
              vm[h][0] = (t0 < lim ? 0x0000ffffu : 0u) | (t0 + 1 < lim ? 0xffff0000u : 0u);
              vm[h][1] = (t0 + 8 < lim ? 0x0000ffffu : 0u) | (t0 + 9 < lim ? 0xffff0000u : 0u);
            }
          }
          // ---- O^T += V^T P^T. Row g of tile dt is output dim 16 g + dt, row g + 8 dim
          // 16 g + 8 + dt (a relabelling of the output dims, undone at the hand-off), so a
          // thread's A operands are bytes of its own 16-code pieces: byte permutes pair the two
          // keys of each operand half (low byte: the even key), which widen exactly to fp16 ----
#pragma unroll
          for (int dp = 0; dp < 4; ++dp) {
            const uint32_t sel = (dp & 1) ? 0x7362u : 0x5140u;   // dims 2 dp, 2 dp + 1
            const int wi = dp >> 1;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint32_t lo01 = __byte_perm(u4_word(vr[h][0], wi), u4_word(vr[h][1], wi), sel);
              const uint32_t hi01 =
                  __byte_perm(u4_word(vr[h][0], wi + 2), u4_word(vr[h][1], wi + 2), sel);
              const uint32_t lo89 = __byte_perm(u4_word(vr[h][2], wi), u4_word(vr[h][3], wi), sel);
              const uint32_t hi89 =
                  __byte_perm(u4_word(vr[h][2], wi + 2), u4_word(vr[h][3], wi + 2), sel);
              uint32_t a0[2], a1[2], a2[2], a3[2];   // [e]: dims 2 dp + e
              e4m3x4_to_f16x4(lo01, a0[0], a0[1]);
              e4m3x4_to_f16x4(hi01, a1[0], a1[1]);
              e4m3x4_to_f16x4(lo89, a2[0], a2[1]);
              e4m3x4_to_f16x4(hi89, a3[0], a3[1]);
#pragma unroll
              for (int e = 0; e < 2; ++e)
                mma_16816(ot[2 * dp + e], a0[e] & vm[h][0], a1[e] & vm[h][0], a2[e] & vm[h][1],
                          a3[e] & vm[h][1], pb[h][0], pb[h][1]);
            }
          }
        }
      } else {
        for (int jj = ((w - j) % NCW + NCW) % NCW; jj < nchunk; jj += NCW) {
          const int gj = j + jj;
          const int st = gj % NST;
          if (RING) {
            if (jj < NCW) rope_prefetch(a, s.c0 + jj, r_lo, lane);   // this warp's first chunk
            if (jj + NCW < nchunk) rope_prefetch(a, s.c0 + jj + NCW, r_lo, lane);
          }
          if (!mbar_wait(bar_full + st * 8, (gj / NST) & 1, abort)) flag_timeout(a, abort);
          const uint32_t stK = sbase + st * L::kStage;
          const uint32_t stV = stK + 2 * kHalfBytes;
          const int c = s.c0 + jj;
          // ring: always masked (the slots' positions are not monotone in the chunk stream)
          const bool full_chunk = !RING && (c + 1) * kChunk <= Lc - a.q_len + 1;
          bool patched = false;
          if (APPEND && (RING || (c + 1) * kChunk > Lc - a.q_len)) {
            const int first_new = Lc - a.q_len;
            const int srow = srow_s[st];
            const uint32_t nkv = sbase + L::newkv_off(a.R, B) + qs * a.q_len * 512;
            const int which = lane >> 4, ch = lane & 15;   // lanes 0-15: K, 16-31: V
            for (int i = 0; i < a.q_len; ++i) {
              const int pos = first_new + i;
              if (pos < 0) continue;
              // the new token's slot in the chunk stream: its position, or its ring slot
              const int slot = !RING ? pos
                             : pos < a.sink ? pos : a.sink + (pos - a.sink) % a.window;
              if (slot < c * kChunk || slot >= (c + 1) * kChunk) continue;
              const int tok = slot - c * kChunk;
              const uint4 val = ld_shared_v4(nkv + i * 512 + which * 256 + ch * 16);
              st_shared_v4((which ? stV : stK) + (ch >> 3) * kHalfBytes + swz128(tok, ch & 7), val);
              if (srow >= 0) {
                __half* pool = which ? a.v_pool : a.k_pool;
                *reinterpret_cast<uint4*>(pool + (static_cast<int64_t>(srow) + tok) * kD + ch * 8) = val;
              }
            }
            __syncwarp();
            patched = true;
          }
          if (RING) {
            rope_pass(a, stK, c, r_lo, lane);
            __syncwarp();
          }
          // ---- S^T = K Q^T: K fragments as the A operand (keys g, g + 8), two chains ----
          float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb2[4] = {0.f, 0.f, 0.f, 0.f};
  #pragma unroll
          for (int sp = 0; sp < 4; ++sp) {
            uint32_t k0[4], k1[4];   // keys 0-7 and 8-15, dims 32 sp .. 32 sp + 31
            const int ch = 4 * sp + (lane >> 3);
            ldsm_x4(stK + (ch >> 3) * kHalfBytes + swz128(lane & 7, ch & 7), k0[0], k0[1], k0[2],
                    k0[3]);
            ldsm_x4(stK + (ch >> 3) * kHalfBytes + swz128(8 + (lane & 7), ch & 7), k1[0], k1[1],
                    k1[2], k1[3]);
            // k-step 2 sp (dims 32 sp .. +15) and 2 sp + 1 (dims 32 sp + 16 .. +31)
            mma_16816(sa, k0[0], k1[0], k0[1], k1[1], qb0[2 * sp], qb1[2 * sp]);
            mma_16816(sb2, k0[2], k1[2], k0[3], k1[3], qb0[2 * sp + 1], qb1[2 * sp + 1]);
          }
          // ---- mask, online softmax over this thread's rows (exp2 domain); the running
          // maximum is brought up to date only when a score exceeds it by more than kLazyLog2 ----
          // sa: [0] key g row 2t4, [1] key g row 2t4+1, [2] key g+8 row 2t4, [3] key g+8 row 2t4+1
          float pv[4];
          float alpha[2] = {1.f, 1.f};
          // positions of keys g and g + 8 (ring: the positions their slots hold)
          const int pos0 = RING ? ring_pos(a, c * kChunk + g, lo_pos, r_lo) : c * kChunk + g;
          const int pos1 = RING ? ring_pos(a, c * kChunk + g + 8, lo_pos, r_lo) : c * kChunk + g + 8;
          float xs[2][2];
          bool grow = false;
  #pragma unroll
          for (int e = 0; e < 2; ++e) {
            float x0 = (sa[e] + sb2[e]) * score_l2;
            float x1 = (sa[2 + e] + sb2[2 + e]) * score_l2;
            if (!full_chunk) {
              x0 = pos0 < tlim[e] ? x0 : kNegInf;
              x1 = pos1 < tlim[e] ? x1 : kNegInf;
            }
            xs[e][0] = x0;
            xs[e][1] = x1;
            grow |= fmaxf(x0, x1) > tm[e] + kLazyLog2;
          }
          if (__any_sync(0xffffffffu, grow)) {
            bool rescale = false;
  #pragma unroll
            for (int e = 0; e < 2; ++e) {
              float mx = fmaxf(xs[e][0], xs[e][1]);
              mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
              mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
              mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
              const float m_old = tm[e];
              const float m_new = fmaxf(m_old, mx);
              const float m_use = m_new == kNegInf ? 0.f : m_new;
              alpha[e] = fast_exp2(m_old - m_use);
              rescale |= (m_old != kNegInf) && (m_new != m_old);
              tm[e] = m_new;
            }
            if (__any_sync(0xffffffffu, rescale)) {
  #pragma unroll
              for (int dt = 0; dt < 8; ++dt) {
                ot[dt][0] *= alpha[0];
                ot[dt][1] *= alpha[1];
                ot[dt][2] *= alpha[0];
                ot[dt][3] *= alpha[1];
              }
            }
          }
  #pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float m_use = tm[e] == kNegInf ? 0.f : tm[e];
            pv[e] = fast_exp2(xs[e][0] - m_use);
            pv[2 + e] = fast_exp2(xs[e][1] - m_use);
            tl[e] = tl[e] * alpha[e] + (pv[e] + pv[2 + e]);
          }
          // P^T (keys x rows) to the B operand (rows g, keys 2t4..): transpose the two 8x8 halves
          const uint32_t pb0 = movmatrix_trans(pack_half2(pv[0], pv[1]));
          const uint32_t pb1 = movmatrix_trans(pack_half2(pv[2], pv[3]));
          // tokens no query may see may hold anything, NaN included: zero their V entries
          uint32_t vm0 = 0xffffffffu, vm1 = 0xffffffffu;
          if (!full_chunk) {
            const int t0 = c * kChunk + 2 * t4;
            if (RING) {
              vm0 = (ring_pos(a, t0, lo_pos, r_lo) < Lc ? 0x0000ffffu : 0u) |
                    (ring_pos(a, t0 + 1, lo_pos, r_lo) < Lc ? 0xffff0000u : 0u);
              vm1 = (ring_pos(a, t0 + 8, lo_pos, r_lo) < Lc ? 0x0000ffffu : 0u) |
                    (ring_pos(a, t0 + 9, lo_pos, r_lo) < Lc ? 0xffff0000u : 0u);
            } else {
              vm0 = (t0 < Lc ? 0x0000ffffu : 0u) | (t0 + 1 < Lc ? 0xffff0000u : 0u);
              vm1 = (t0 + 8 < Lc ? 0x0000ffffu : 0u) | (t0 + 9 < Lc ? 0xffff0000u : 0u);
            }
          }
          // ---- O^T += V^T P^T: V fragments as the A operand ----
  #pragma unroll
          for (int dt = 0; dt < 8; ++dt) {
            const int i = lane >> 3;
            const int tok = (i & 1) * 8 + (lane & 7);
            const int ch = 2 * dt + (i >> 1);
            uint32_t v0, v1, v2, v3;
            ldsm_x4_trans(stV + (ch >> 3) * kHalfBytes + swz128(tok, ch & 7), v0, v1, v2, v3);
            v0 &= vm0; v1 &= vm1; v2 &= vm0; v3 &= vm1;
            mma_16816(ot[dt], v0, v2, v1, v3, pb0, pb1);
          }
          if (RING || (APPEND && patched)) fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_empty + st * 8);
        }
      }
      if (kHoldQ) {
        if (RING) fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_qempty + qs * 8);
      }
      j += FP8 ? (nchunk + 1) >> 1 : nchunk;   // stages of the segment
      // ---- hand this warp's state to the epilogue: rows 2t4, 2t4 + 1 ----
      const int sb = k & 1;
      if (k >= 2 && !mbar_wait(bar_sfree + sb * 8, ((k >> 1) - 1) & 1, abort)) flag_timeout(a, abort);
      float* o_d = stO + sb * NCW * a.R * kSt;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float lv = tl[e];
        lv += __shfl_xor_sync(0xffffffffu, lv, 4);
        lv += __shfl_xor_sync(0xffffffffu, lv, 8);
        lv += __shfl_xor_sync(0xffffffffu, lv, 16);
        const int r = 2 * t4 + e;
        if (r < a.R) {
          float* row = o_d + (w * a.R + r) * kSt;
          if constexpr (FP8) {
            // dims 16 g + dt (tile rows g) and 16 g + 8 + dt (rows g + 8), scaled by the V scale
            float4* dst = reinterpret_cast<float4*>(row + 16 * g);
            dst[0] = make_float4(ot[0][e] * out_sc, ot[1][e] * out_sc, ot[2][e] * out_sc, ot[3][e] * out_sc);
            dst[1] = make_float4(ot[4][e] * out_sc, ot[5][e] * out_sc, ot[6][e] * out_sc, ot[7][e] * out_sc);
            dst[2] = make_float4(ot[0][2 + e] * out_sc, ot[1][2 + e] * out_sc, ot[2][2 + e] * out_sc,
                                 ot[3][2 + e] * out_sc);
            dst[3] = make_float4(ot[4][2 + e] * out_sc, ot[5][2 + e] * out_sc, ot[6][2 + e] * out_sc,
                                 ot[7][2 + e] * out_sc);
          } else {
#pragma unroll
            for (int dt = 0; dt < 8; ++dt) {
              row[g + 16 * dt] = ot[dt][e];
              row[g + 16 * dt + 8] = ot[dt][2 + e];
            }
          }
          if (g == 0) {
            stM[(sb * NCW + w) * a.R + r] = tm[e];
            stL[(sb * NCW + w) * a.R + r] = lv;
          }
        }
      }
      } else {
      // Q fragments (A operand, 16 rows x 128 dims per m-tile)
      uint32_t qf[MT == 1 ? 8 : 1][4];
      auto q_frag = [&](int mt, int s8, uint32_t (&f)[4]) {
        const int i = lane >> 3;
        const int row = mt * 16 + (i & 1) * 8 + (lane & 7);
        const int ch = 2 * s8 + (i >> 1);
        ldsm_x4(qb + (ch >> 3) * L::kQHalf + swz128(row, ch & 7), f[0], f[1], f[2], f[3]);
      };
      if (MT == 1) {
#pragma unroll
        for (int s8 = 0; s8 < 8; ++s8) q_frag(0, s8, qf[s8]);
        if (!kHoldQ) {
          if (RING) fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_qempty + qs * 8);
        }
      }

      float m_run[MT][2], l_run[MT][2], o[MT][16][4];
  #pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        m_run[mt][0] = m_run[mt][1] = kNegInf;
        l_run[mt][0] = l_run[mt][1] = 0.f;
  #pragma unroll
        for (int nd = 0; nd < 16; ++nd) o[mt][nd][0] = o[mt][nd][1] = o[mt][nd][2] = o[mt][nd][3] = 0.f;
      }
      // causal limit of each of this thread's rows: query qi sees positions < Lc - q_len + qi + 1
      int lim[MT][2];
  #pragma unroll
      for (int mt = 0; mt < MT; ++mt)
  #pragma unroll
        for (int rh = 0; rh < 2; ++rh) {
          const int r = mt * 16 + rh * 8 + g;
          const int qi = r < a.R ? r / a.G : a.q_len - 1;
          lim[mt][rh] = Lc - a.q_len + qi + 1;
        }

      const int nchunk = s.c1 - s.c0;
      // this warp's chunks of the segment: CTA-local index j + jj with (j + jj) % NCW == w
      for (int jj = ((w - j) % NCW + NCW) % NCW; jj < nchunk; jj += NCW) {
        const int gj = j + jj;
        const int st = gj % NST;
        if (RING) {
          if (jj < NCW) rope_prefetch(a, s.c0 + jj, r_lo, lane);   // this warp's first chunk
          if (jj + NCW < nchunk) rope_prefetch(a, s.c0 + jj + NCW, r_lo, lane);
        }
        if (!mbar_wait(bar_full + st * 8, (gj / NST) & 1, abort)) flag_timeout(a, abort);
        const uint32_t stK = sbase + st * kStageBytes;
        const uint32_t stV = stK + 2 * kHalfBytes;
        const int c = s.c0 + jj;

        // positions of this thread's score columns (tokens nt*8 + 2*t4 + e) and of its K rows
        int pcol[2][2];
  #pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
  #pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int t = c * kChunk + nt * 8 + 2 * t4 + e;
            if (!RING) {
              pcol[nt][e] = t;
            } else {
              int p;
              if (t < a.sink) p = t;
              else if (t < cap) { int d = t - r_lo; if (d < 0) d += a.window; p = lo_pos + d; }
              else p = 0x7fffffff;
              pcol[nt][e] = p;
            }
          }
        }
        // whole chunk visible to every query row?
        bool full_chunk;
        if (!RING) full_chunk = (c + 1) * kChunk <= Lc - a.q_len + 1;
        else full_chunk = false;

        // ---- fused append: this chunk holds some of the step's new tokens (the last q_len
        // positions of the sequence). Their K/V rows, loaded with the segment's queries, replace
        // the stale slots in the landed tile and are written to the pool (the chunk's TMA row
        // plus the token's offset: the slot the table maps that position to). ----
        bool patched = false;
        if (APPEND && (RING || (c + 1) * kChunk > Lc - a.q_len)) {
          const int first_new = Lc - a.q_len;
          const int srow = srow_s[st];
          const uint32_t nkv = sbase + L::newkv_off(a.R, B) + qs * a.q_len * 512;
          const int which = lane >> 4, ch = lane & 15;   // lanes 0-15: K, 16-31: V
          for (int i = 0; i < a.q_len; ++i) {
            const int pos = first_new + i;
            if (pos < 0) continue;
            // the new token's slot in the chunk stream: its position (paged), or its ring slot
            // Slot(pos) (sink + ring)
            const int slot = !RING ? pos
                           : pos < a.sink ? pos : a.sink + (pos - a.sink) % a.window;
            if (slot < c * kChunk || slot >= (c + 1) * kChunk) continue;
            const int tok = slot - c * kChunk;
            const uint4 val = ld_shared_v4(nkv + i * 512 + which * 256 + ch * 16);
            st_shared_v4((which ? stV : stK) + (ch >> 3) * kHalfBytes + swz128(tok, ch & 7), val);
            if (srow >= 0) {
              __half* pool = which ? a.v_pool : a.k_pool;
              *reinterpret_cast<uint4*>(pool + (static_cast<int64_t>(srow) + tok) * kD + ch * 8) = val;
            }
          }
          __syncwarp();
          patched = true;
        }

        if (RING) {
          rope_pass(a, stK, c, r_lo, lane);
          __syncwarp();
        }

        // ---- S = Q K^T ----
        // K fragments of both 8-token halves first, then two independent accumulator chains
        // per half (even / odd k-steps) so that consecutive mma do not wait on each other.
        uint32_t kf[2][8][2];
  #pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
  #pragma unroll
          for (int sp = 0; sp < 4; ++sp) {
            const int ch = 4 * sp + (lane >> 3);
            const int tok = nt * 8 + (lane & 7);
            ldsm_x4(stK + (ch >> 3) * kHalfBytes + swz128(tok, ch & 7), kf[nt][2 * sp][0],
                    kf[nt][2 * sp][1], kf[nt][2 * sp + 1][0], kf[nt][2 * sp + 1][1]);
          }
        }
        // two accumulator chains per m-tile (even / odd k-steps) for one m-tile; two m-tiles
        // already give two independent chains
        constexpr bool kDual = MT == 1;
        float sc[MT][2][4], sc2[kDual ? MT : 1][2][4];
  #pragma unroll
        for (int mt = 0; mt < MT; ++mt)
  #pragma unroll
          for (int nt = 0; nt < 2; ++nt)
  #pragma unroll
            for (int i = 0; i < 4; ++i) {
              sc[mt][nt][i] = 0.f;
              if (kDual) sc2[kDual ? mt : 0][nt][i] = 0.f;
            }
  #pragma unroll
        for (int mt = 0; mt < MT; ++mt)
  #pragma unroll
          for (int s8 = 0; s8 < 8; ++s8) {
            uint32_t f[4];
            if (MT == 1) {
              f[0] = qf[s8][0]; f[1] = qf[s8][1]; f[2] = qf[s8][2]; f[3] = qf[s8][3];
            } else {
              q_frag(mt, s8, f);
            }
  #pragma unroll
            for (int nt = 0; nt < 2; ++nt)
              mma_16816((kDual && (s8 & 1)) ? sc2[kDual ? mt : 0][nt] : sc[mt][nt], f[0], f[1],
                        f[2], f[3], kf[nt][s8][0], kf[nt][s8][1]);
          }

        // ---- mask, online softmax (exp2 domain); a row's running maximum is brought up to
        // date only when one of its scores exceeds it by more than kLazyLog2 ----
        uint32_t pa[MT][4];
        float alpha[MT][2];
        float v[MT][2][4];
        bool grow = false;
  #pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
  #pragma unroll
          for (int rh = 0; rh < 2; ++rh) {
            alpha[mt][rh] = 1.f;
  #pragma unroll
            for (int nt = 0; nt < 2; ++nt)
  #pragma unroll
              for (int e = 0; e < 2; ++e) {
                const float x = (kDual ? sc[mt][nt][rh * 2 + e] + sc2[kDual ? mt : 0][nt][rh * 2 + e]
                                       : sc[mt][nt][rh * 2 + e]) * a.scale_log2;
                v[mt][rh][nt * 2 + e] = (full_chunk || pcol[nt][e] < lim[mt][rh]) ? x : kNegInf;
              }
            const float lm = fmaxf(fmaxf(v[mt][rh][0], v[mt][rh][1]), fmaxf(v[mt][rh][2], v[mt][rh][3]));
            grow |= lm > m_run[mt][rh] + kLazyLog2;
          }
        }
        if (__any_sync(0xffffffffu, grow)) {
          bool rescale = false;
  #pragma unroll
          for (int mt = 0; mt < MT; ++mt)
  #pragma unroll
            for (int rh = 0; rh < 2; ++rh) {
              float mx = fmaxf(fmaxf(v[mt][rh][0], v[mt][rh][1]), fmaxf(v[mt][rh][2], v[mt][rh][3]));
              mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
              mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
              const float m_old = m_run[mt][rh];
              const float m_new = fmaxf(m_old, mx);
              const float m_use = m_new == kNegInf ? 0.f : m_new;
              // O and l are still exactly zero while m_old is -inf, so only a finite, grown
              // maximum needs the accumulators rescaled
              alpha[mt][rh] = fast_exp2(m_old - m_use);
              rescale |= (m_old != kNegInf) && (m_new != m_old);
              m_run[mt][rh] = m_new;
            }
          if (__any_sync(0xffffffffu, rescale)) {
  #pragma unroll
            for (int mt = 0; mt < MT; ++mt)
  #pragma unroll
              for (int nd = 0; nd < 16; ++nd) {
                o[mt][nd][0] *= alpha[mt][0];
                o[mt][nd][1] *= alpha[mt][0];
                o[mt][nd][2] *= alpha[mt][1];
                o[mt][nd][3] *= alpha[mt][1];
              }
          }
        }
  #pragma unroll
        for (int mt = 0; mt < MT; ++mt)
  #pragma unroll
          for (int rh = 0; rh < 2; ++rh) {
            const float m_use = m_run[mt][rh] == kNegInf ? 0.f : m_run[mt][rh];
            float rs = 0.f;
  #pragma unroll
            for (int i = 0; i < 4; ++i) {
              v[mt][rh][i] = fast_exp2(v[mt][rh][i] - m_use);
              rs += v[mt][rh][i];
            }
            l_run[mt][rh] = l_run[mt][rh] * alpha[mt][rh] + rs;
            // P as the A operand: a0/a2 hold row g, a1/a3 row g+8
            pa[mt][rh] = pack_half2(v[mt][rh][0], v[mt][rh][1]);
            pa[mt][2 + rh] = pack_half2(v[mt][rh][2], v[mt][rh][3]);
          }

        // tokens no query may see (past the cache, or not in the ring's valid set) may hold
        // anything, NaN included: zero their V entries so that 0 * V stays 0
        uint32_t vm0 = 0xffffffffu, vm1 = 0xffffffffu;
        if (!full_chunk) {
          const int all = Lc;  // the last query's limit
          vm0 = (pcol[0][0] < all ? 0x0000ffffu : 0u) | (pcol[0][1] < all ? 0xffff0000u : 0u);
          vm1 = (pcol[1][0] < all ? 0x0000ffffu : 0u) | (pcol[1][1] < all ? 0xffff0000u : 0u);
        }

        // ---- O += P V ----
  #pragma unroll
        for (int np = 0; np < 8; ++np) {
          const int i = lane >> 3;
          const int tok = (i & 1) * 8 + (lane & 7);
          const int ch = 2 * np + (i >> 1);
          uint32_t v0, v1, v2, v3;
          ldsm_x4_trans(stV + (ch >> 3) * kHalfBytes + swz128(tok, ch & 7), v0, v1, v2, v3);
          v0 &= vm0; v1 &= vm1; v2 &= vm0; v3 &= vm1;
  #pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            mma_16816(o[mt][2 * np], pa[mt][0], pa[mt][1], pa[mt][2], pa[mt][3], v0, v1);
            mma_16816(o[mt][2 * np + 1], pa[mt][0], pa[mt][1], pa[mt][2], pa[mt][3], v2, v3);
          }
        }
        // a patched (or, ring, rotated) tile was written through the generic proxy; order that
        // before the next TMA (async proxy) write into this stage
        if (RING || (APPEND && patched)) fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_empty + st * 8);
      }
      if (kHoldQ) {
        if (RING) fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_qempty + qs * 8);
      }
      j += nchunk;

      // ---- hand this warp's state for the segment to the epilogue warp ----
      const int sb = k & 1;
      if (k >= 2 && !mbar_wait(bar_sfree + sb * 8, ((k >> 1) - 1) & 1, abort)) flag_timeout(a, abort);
      float* o_d = stO + sb * NCW * a.R * kSt;
  #pragma unroll
      for (int mt = 0; mt < MT; ++mt)
  #pragma unroll
        for (int rh = 0; rh < 2; ++rh) {
          float lv = l_run[mt][rh];
          lv += __shfl_xor_sync(0xffffffffu, lv, 1);
          lv += __shfl_xor_sync(0xffffffffu, lv, 2);
          const int r = mt * 16 + rh * 8 + g;
          if (r < a.R) {
            float* dst = o_d + (w * a.R + r) * kSt + 2 * t4;
  #pragma unroll
            for (int nd = 0; nd < 16; ++nd)
              *reinterpret_cast<float2*>(dst + nd * 8) = make_float2(o[mt][nd][rh * 2], o[mt][nd][rh * 2 + 1]);
            if (t4 == 0) {
              stM[(sb * NCW + w) * a.R + r] = m_run[mt][rh];
              stL[(sb * NCW + w) * a.R + r] = lv;
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_sdone + (k & 1) * 8);
      ++k;
      has = cur.next(s);
    }
  }

  // ---- end of the slice: consumers and epilogue merge the last segment, then any split unit
  // whose last partial arrived from this CTA (the producer has left)
  if (warp != NCW && last_k >= 0) {
    const int t = warp < NCW ? tid : tid - 32;   // dense index over consumers + epilogue
    const int ua = unit_first(pre, a.Hkv, last_b, last_h, last_nb);
    const int parts = (ua + last_nb - 1) / per - ua / per + 1;
    const MergeStage ms(smem, L::kQ, a.R);
    named_barrier_sync(2, kNE);                  // last states written, earlier segments merged
    const int sb = last_k & 1;
    float* so_w = stO + sb * NCW * a.R * kSt;
    const float* sm_w = stM + sb * NCW * a.R;
    const float* sl_w = stL + sb * NCW * a.R;
    int* counter = a.counters + last_b * a.Hkv + last_h;
    // A split unit is merged by the CTA that holds its first chunk, the one whose last segment
    // is the unit's head. That CTA keeps its own partial in the staging area (it never goes out
    // to the workspace and back) and waits until the other CTAs have announced theirs; most of
    // them finished that work long before (a unit's other parts are the first segments of
    // later CTAs, or whole slices). The wait is bounded in time: if the other parts are not in
    // (their CTAs may not be resident yet, e.g. when other work holds the GPU), the CTA
    // announces its partial like the others and the last to arrive merges. Either way the
    // partials and their order are the same, so the result does not depend on the path.
    bool merged = false;
    if (!last_complete && last_head) {
      merge_segment_wide<NCW, kNE>(a, so_w, sm_w, sl_w, last_b, last_h, false, ms.so, ms.sml,
                                   t);
      if (t == 0) {
        const uint64_t t_end = global_time_ns() + kMergeWaitNs;
        int ok = 0;
        do {
          if (ld_acquire_gpu(counter) == parts - 1) { ok = 1; break; }
        } while (global_time_ns() < t_end);
        *fast_s = ok;
      }
      named_barrier_sync(2, kNE);
      merged = *fast_s;
      if (merged) {
        merge_unit<kNE>(a, last_b, last_h, last_nb, pre, per, smem, L::kQ, t,
                        blockIdx.x);
      } else {
        // give up waiting: the staged partial goes to the workspace like the others'
        float* po = a.part_o + static_cast<int64_t>(last_slot) * a.R * kD;
        float* pml = a.part_ml + static_cast<int64_t>(last_slot) * a.R * 4;
        for (int i = t; i < a.R * 32; i += kNE)
          reinterpret_cast<float4*>(po)[i] = reinterpret_cast<const float4*>(ms.so)[i];
        if (t < a.R) reinterpret_cast<float4*>(pml)[t] = reinterpret_cast<const float4*>(ms.sml)[t];
      }
    } else {
      merge_segment_wide<NCW, kNE>(a, so_w, sm_w, sl_w, last_b, last_h, last_complete,
                                   a.part_o + static_cast<int64_t>(last_slot) * a.R * kD,
                                   a.part_ml + static_cast<int64_t>(last_slot) * a.R * 4, t);
    }
    if (!last_complete && !merged) {
      named_barrier_sync(2, kNE);                // partial written by every thread
      if (t == 0 && atomic_add_acq_rel(counter, 1) == parts - 1) {
        const int n = *npend_s;
        npend_s[1 + 3 * n] = last_b;
        npend_s[2 + 3 * n] = last_h;
        npend_s[3 + 3 * n] = last_nb;
        *npend_s = n + 1;
      }
    }
    named_barrier_sync(2, kNE);
    const int np = *npend_s;
    // every chunk of this CTA's slice has been consumed, so the stage memory is free
#pragma unroll 1
    for (int i = 0; i < np; ++i)
      merge_unit<kNE>(a, npend_s[1 + 3 * i], npend_s[2 + 3 * i], npend_s[3 + 3 * i], pre, per,
                      smem, L::kQ, t);
  }
}

// ---------------------------------------------------------------------------------------------
// Host side.

// Consumer warps and stages per CTA. The paged kernels stream: two consumer warps keep up
// with HBM, and the shared memory goes to stages. The ring kernels rotate every key (RoPE on
// read) and are bound by the consumers' arithmetic: four consumer warps, eight stages.
constexpr int kNCW = PKV_DECODE_WARPS, kNST = PKV_DECODE_STAGES;
constexpr int kNCWRing = 4, kNSTRing = 8;
// The ring's transposed-tile kernels (up to 8 rows): their per-chunk RoPE pass is a chain of
// dependent shared-memory and arithmetic steps, so more consumer warps per SM hide more of
// it: two CTAs of four consumer warps and eight stages each (eight per SM; one CTA of six
// warps and twelve stages measured 1.7 % slower on the ring step).
#ifndef PKV_RING_TR_WARPS
#define PKV_RING_TR_WARPS 4
#endif
#ifndef PKV_RING_TR_STAGES
#define PKV_RING_TR_STAGES 8
#endif
constexpr int kNCWRingTR = PKV_RING_TR_WARPS, kNSTRingTR = PKV_RING_TR_STAGES;
// The E4M3 cache: 8 KB stages of two chunks each (the producer's per-stage work, and the
// consumers' per-softmax-step work, spread over twice the keys of an fp16 stage's bytes), two
// CTAs per SM. Widening the codes adds to each consumer warp's work, so four consumer warps
// share the stages (eight stages, 64 KB of K/V in flight per CTA).
#ifndef PKV_FP8_WARPS
#define PKV_FP8_WARPS 4
#endif
#ifndef PKV_FP8_STAGES
#define PKV_FP8_STAGES 8
#endif
constexpr int kNCWFp8 = PKV_FP8_WARPS, kNSTFp8 = PKV_FP8_STAGES;

using KernelFn = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, DecodeArgs);

// Whether the fused-append calls may start while the kernel before them finishes
// (programmatic dependent launch); process-wide, read at each launch.
std::atomic<int> g_early_start{1};

struct Variant {
  const void* fn;
  int mt;
  bool ring;
  int threads;
  size_t (*smem)(int R, int B, int newkv_bytes);
};

template <int NCW, int NST, int MT, bool FP8 = false>
size_t smem_of(int R, int B, int newkv_bytes) {
  return Smem<NCW, NST, MT, FP8>::bytes(R, B, newkv_bytes);
}

template <int MT, bool RING, bool APPEND, bool TR = false, bool FP8 = false, bool KV3D = false>
Variant variant() {
  constexpr int NCW = RING ? (TR ? kNCWRingTR : kNCWRing) : FP8 ? kNCWFp8 : kNCW;
  constexpr int NST = RING ? (TR ? kNSTRingTR : kNSTRing) : FP8 ? kNSTFp8 : kNST;
  return Variant{
      reinterpret_cast<const void*>(&decode_kernel<NCW, NST, MT, RING, APPEND, TR, FP8, KV3D>), MT,
      RING, (NCW + 2) * 32, &smem_of<NCW, NST, MT, FP8>};
}

// Persistent grid for a variant: SM count x resident CTAs (capped), cached per device/size.
int grid_size(const Variant& v, size_t smem, int* status) {
  static std::mutex mu;
  static std::map<std::tuple<int, const void*, size_t>, int> cache;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) { *status = cuda_status(e); return 0; }
  std::lock_guard<std::mutex> lock(mu);
  auto key = std::make_tuple(dev, v.fn, smem);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  // The attribute is per kernel, not per launch: raise it once to the device's limit, so that
  // a launch with a smaller size never lowers it under a later, larger one (whose grid is
  // already cached).
  int limit = 0;
  e = cudaDeviceGetAttribute(&limit, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e == cudaSuccess && static_cast<size_t>(limit) < smem) e = cudaErrorInvalidValue;
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(v.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, limit);
  int occ = 0;
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, v.fn, v.threads, smem);
  if (e != cudaSuccess) { *status = cuda_status(e); return 0; }
  if (occ < 1) { *status = PKV_EINVAL; return 0; }
  const int grid = sm_count() * std::min(occ, kMaxCtasPerSm);
  cache[key] = grid;
  return grid;
}

struct WsLayout {
  size_t counters, part_ml, part_o, total;
};

WsLayout ws_layout(int num_seqs, int Hkv, int R) {
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  const size_t partials = static_cast<size_t>(2) * sm_count() * kMaxCtasPerSm;
  WsLayout w;
  w.counters = 0;
  w.part_ml = up(static_cast<size_t>(num_seqs) * Hkv * sizeof(int));
  w.part_o = w.part_ml + up(partials * R * 4 * sizeof(float));
  w.total = w.part_o + up(partials * R * kD * sizeof(float));
  return w;
}

int encode(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims,
           const cuuint64_t* strides, const cuuint32_t* box,
           CUtensorMapDataType type = CU_TENSOR_MAP_DATA_TYPE_FLOAT16) {
  auto fn = tensor_map_encoder();
  if (!fn) return PKV_ECUDA_BASE - static_cast<int>(cudaErrorNotSupported);
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, type, rank, const_cast<void*>(base), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PKV_OK : PKV_EINVAL;
}

int launch_decode(bool ring, void* out, const void* q, const void* k_new, const void* v_new,
                  const void* k_cache, const void* v_cache,
                  int num_blocks, const int32_t* block_tables, int max_blocks,
                  const int32_t* context_lens, const int64_t* logical_len,
                  const int64_t* high_water, int num_seqs, int q_len, int Hq, int Hkv,
                  int head_dim, int block_size, int sink, int window, const float* rope,
                  float scale, void* workspace, size_t workspace_bytes, pkv_stream_t stream,
                  const float* k_scale = nullptr, const float* v_scale = nullptr) {
  if (num_seqs < 0 || q_len < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || head_dim != kD ||
      !valid_block_size(block_size) || num_blocks < 0 || max_blocks < 0)
    return PKV_EINVAL;
  if (num_seqs == 0) return PKV_OK;
  if (num_seqs > kMaxSeqs) return PKV_EINVAL;
  const int G = Hq / Hkv;
  const int R = G * q_len;
  if (R > 32) return PKV_EINVAL;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !workspace) return PKV_EINVAL;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return PKV_EINVAL;
  const bool append = k_new != nullptr;
  if (append && (!v_new || !aligned16(k_new) || !aligned16(v_new))) return PKV_EINVAL;
  // the new tokens of one call must land in distinct ring slots
  if (append && ring && q_len > window) return PKV_EINVAL;
  const bool fp8 = k_scale != nullptr;
  if (fp8 && (ring || !v_scale || G * q_len > 8)) return PKV_EINVAL;
  if (ring) {
    if (!logical_len || !high_water || !rope || sink < 0 || window < 1) return PKV_EINVAL;
    if ((sink + window + block_size - 1) / block_size > max_blocks) return PKV_EINVAL;
  } else if (!context_lens) {
    return PKV_EINVAL;
  }
  // all chunk indices and TMA rows fit in int32
  const int64_t rows = static_cast<int64_t>(num_blocks) * Hkv * block_size;
  const int64_t max_ctx = ring ? (sink + window) : static_cast<int64_t>(max_blocks) * block_size;
  if (rows >= (1ll << 31) || static_cast<int64_t>(num_seqs) * Hkv * ((max_ctx + kChunk - 1) / kChunk + kSegCost) >= (1ll << 30))
    return PKV_EINVAL;
  if (num_blocks == 0) return PKV_EINVAL;
  const WsLayout ws = ws_layout(num_seqs, Hkv, R);
  if (workspace_bytes < ws.total) return PKV_ENOSPC;

  const int mt = R <= 16 ? 1 : 2;
  // up to 8 rows per unit (GQA groups of 6-8 at one query token): the transposed tile
  const bool tr = R <= 8;
  // With one query row per unit (MHA, paged) a chunk's consumer work is light and the stream is
  // bound by the producer's issue rate: two 3-D boxes per chunk instead of four 2-D ones
  // measured 20 % faster on an MHA batch whose shared prefix hits L2 (2.5 % without sharing).
  // With grouped heads the 2-D boxes measured faster (up to 2.6 %), so they stay there.
  const bool kv3d = !fp8 && !ring && G == 1 && tr;
  Variant v = fp8      ? (append ? variant<1, false, true, true, true>()
                                 : variant<1, false, false, true, true>())
              : kv3d   ? (append ? variant<1, false, true, true, false, true>()
                                 : variant<1, false, false, true, false, true>())
              : ring   ? (append ? (tr ? variant<1, true, true, true>()
                                         : mt == 1 ? variant<1, true, true>() : variant<2, true, true>())
                                 : (tr ? variant<1, true, false, true>()
                                       : mt == 1 ? variant<1, true, false>() : variant<2, true, false>()))
              : append ? (tr ? variant<1, false, true, true>()
                             : mt == 1 ? variant<1, false, true>() : variant<2, false, true>())
                       : (tr ? variant<1, false, false, true>()
                             : mt == 1 ? variant<1, false, false>() : variant<2, false, false>());
  const int newkv_bytes = append ? 2 * q_len * 512 : 0;
  const size_t smem = v.smem(R, num_seqs, newkv_bytes);
  if (smem > 227 * 1024) return PKV_EINVAL;
  int status = PKV_OK;
  const int grid = grid_size(v, smem, &status);
  if (!grid) return status != PKV_OK ? status : PKV_EINVAL;

  CUtensorMap tmK, tmV, tmQ;
  int st;
  if (fp8) {
    // rows of 128 E4M3 bytes: one 16-row box per chunk
    const cuuint64_t kv_dims[2] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(rows)};
    const cuuint64_t kv_strides[1] = {static_cast<cuuint64_t>(kD)};
    const cuuint32_t kv_box[2] = {static_cast<cuuint32_t>(kD), kChunk};
    st = encode(&tmK, k_cache, 2, kv_dims, kv_strides, kv_box, CU_TENSOR_MAP_DATA_TYPE_UINT8);
    if (st == PKV_OK)
      st = encode(&tmV, v_cache, 2, kv_dims, kv_strides, kv_box, CU_TENSOR_MAP_DATA_TYPE_UINT8);
  } else if (kv3d) {
    // rows of 128 fp16 seen as (64 columns, rows, 2 halves of 64 columns): one box of
    // 64 x 16 x 2 brings a chunk's two 64-column halves, one after the other, each a
    // 128-byte-swizzled 2 KB tile as the fragment loads expect
    const cuuint64_t kv_dims[3] = {64, static_cast<cuuint64_t>(rows), 2};
    const cuuint64_t kv_strides[2] = {kD * 2, 64 * 2};
    const cuuint32_t kv_box[3] = {64, kChunk, 2};
    st = encode(&tmK, k_cache, 3, kv_dims, kv_strides, kv_box);
    if (st == PKV_OK) st = encode(&tmV, v_cache, 3, kv_dims, kv_strides, kv_box);
  } else {
    // rows of 128 fp16: a 64 x 16 box per 64-column half of a chunk
    const cuuint64_t kv_dims[2] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(rows)};
    const cuuint64_t kv_strides[1] = {kD * 2};
    const cuuint32_t kv_box[2] = {64, kChunk};
    st = encode(&tmK, k_cache, 2, kv_dims, kv_strides, kv_box);
    if (st == PKV_OK) st = encode(&tmV, v_cache, 2, kv_dims, kv_strides, kv_box);
  }
  const cuuint64_t q_dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(Hq),
                                static_cast<cuuint64_t>(num_seqs) * q_len};
  const cuuint64_t q_strides[2] = {kD * 2, static_cast<cuuint64_t>(Hq) * kD * 2};
  const cuuint32_t q_box[3] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(q_len)};
  if (st == PKV_OK) st = encode(&tmQ, q, 3, q_dims, q_strides, q_box);
  if (st != PKV_OK) return st;

  unsigned int* err = device_error_ptr();
  if (!err) return cuda_status(cudaGetLastError());
  DecodeArgs args;
  args.out = static_cast<__half*>(out);
  args.block_tables = block_tables;
  args.context_lens = context_lens;
  args.logical_len = logical_len;
  args.high_water = high_water;
  args.rope = rope;
  uint8_t* wsb = static_cast<uint8_t*>(workspace);
  args.counters = reinterpret_cast<int*>(wsb + ws.counters);
  args.part_ml = reinterpret_cast<float*>(wsb + ws.part_ml);
  args.part_o = reinterpret_cast<float*>(wsb + ws.part_o);
  args.err = err;
  args.num_blocks = num_blocks;
  args.max_blocks = max_blocks;
  args.num_seqs = num_seqs;
  args.q_len = q_len;
  args.Hq = Hq;
  args.Hkv = Hkv;
  args.G = G;
  args.R = R;
  args.block_size = block_size;
  int shift = 0;
  while ((kChunk << shift) < block_size) ++shift;
  args.bs_shift = shift;
  args.sink = sink;
  args.window = window;
  args.scale_log2 = scale * 1.4426950408889634f;
  args.k_new = static_cast<const __half*>(k_new);
  args.v_new = static_cast<const __half*>(v_new);
  args.k_pool = static_cast<__half*>(const_cast<void*>(k_cache));
  args.v_pool = static_cast<__half*>(const_cast<void*>(v_cache));
  args.k_scale = k_scale;
  args.v_scale = v_scale;

  void* params[4] = {&tmK, &tmV, &tmQ, &args};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(v.threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = static_cast<cudaStream_t>(stream);
  // the fused-append call may start while the preceding kernel finishes (see the kernel)
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = (append && g_early_start.load(std::memory_order_relaxed)) ? 1 : 0;
  return cuda_status(cudaLaunchKernelExC(&cfg, v.fn, params));
}

// ---------------------------------------------------------------------------------------------
// Decode without caller-provided scratch. Some callers cannot allocate device memory at all:
// code running under a caller that owns every device allocation (a host framework's plugin
// interface, an embedded runtime with a fixed memory budget), or code that must not enter an
// allocator at the point where it runs. For them the decode's scratch (arrival counters and
// split-context partials) lives in this fixed array instead. Every GPU that loads the library
// holds it until the process exits.
constexpr size_t kFixedScratchBytes = size_t(8) << 20;   // 8 MiB
static __device__ __align__(256) unsigned char g_decode_scratch[kFixedScratchBytes];

// Device address of g_decode_scratch on the current device. In host code the array's name is
// only a host-side stand-in, so the address is resolved once per device (with that device
// current) and cached.
void* fixed_scratch(int* status) {
  static std::mutex mu;
  static void* ptrs[64] = {};
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) { *status = cuda_status(e); return nullptr; }
  if (dev < 0 || dev >= 64) { *status = PKV_EINVAL; return nullptr; }
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) { *status = cuda_status(e); return nullptr; }
    ptrs[dev] = p;
  }
  return ptrs[dev];
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" {

size_t pkv_decode_workspace_bytes(int num_seqs, int q_len, int num_q_heads, int num_kv_heads,
                                  int head_dim) {
  if (num_seqs < 0 || q_len < 1 || num_q_heads < 1 || num_kv_heads < 1 ||
      num_q_heads % num_kv_heads || head_dim != kD || sm_count() == 0)
    return 0;
  const int R = num_q_heads / num_kv_heads * q_len;
  return ws_layout(std::max(num_seqs, 1), num_kv_heads, R).total;
}

int pkv_set_early_start(int enable) {
  return g_early_start.exchange(enable != 0 ? 1 : 0);
}

int pkv_workspace_init(void* workspace, size_t workspace_bytes, pkv_stream_t stream) {
  if (!workspace) return PKV_EINVAL;
  return cuda_status(cudaMemsetAsync(workspace, 0, workspace_bytes,
                                     static_cast<cudaStream_t>(stream)));
}

int pkv_paged_attn_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                          int num_blocks, const int32_t* block_tables, int max_blocks_per_seq,
                          const int32_t* context_lens, int num_seqs, int q_len, int num_q_heads,
                          int num_kv_heads, int head_dim, int block_size, float scale,
                          void* workspace, size_t workspace_bytes, pkv_stream_t stream) {
  return launch_decode(false, out, q, nullptr, nullptr, k_cache, v_cache, num_blocks, block_tables,
                       max_blocks_per_seq, context_lens, nullptr, nullptr, num_seqs, q_len,
                       num_q_heads, num_kv_heads, head_dim, block_size, 0, 1, nullptr, scale,
                       workspace, workspace_bytes, stream);
}

int pkv_paged_attn_decode_append_fp8(void* out, const void* q, const void* k_new,
                                     const void* v_new, void* k_cache, void* v_cache,
                                     const float* k_scale, const float* v_scale, int num_blocks,
                                     const int32_t* block_tables, int max_blocks_per_seq,
                                     const int32_t* context_lens, int num_seqs, int q_len,
                                     int num_q_heads, int num_kv_heads, int head_dim,
                                     int block_size, float scale, void* workspace,
                                     size_t workspace_bytes, pkv_stream_t stream) {
  if (!k_scale || !v_scale || (num_seqs > 0 && (!k_new || !v_new))) return PKV_EINVAL;
  return launch_decode(false, out, q, num_seqs > 0 ? k_new : nullptr, v_new, k_cache, v_cache,
                       num_blocks, block_tables, max_blocks_per_seq, context_lens, nullptr,
                       nullptr, num_seqs, q_len, num_q_heads, num_kv_heads, head_dim,
                       block_size, 0, 1, nullptr, scale, workspace, workspace_bytes, stream,
                       k_scale, v_scale);
}

int pkv_paged_attn_decode_fp8(void* out, const void* q, const void* k_cache,
                              const void* v_cache, const float* k_scale, const float* v_scale,
                              int num_blocks, const int32_t* block_tables,
                              int max_blocks_per_seq, const int32_t* context_lens, int num_seqs,
                              int q_len, int num_q_heads, int num_kv_heads, int head_dim,
                              int block_size, float scale, void* workspace,
                              size_t workspace_bytes, pkv_stream_t stream) {
  if (!k_scale || !v_scale) return PKV_EINVAL;
  return launch_decode(false, out, q, nullptr, nullptr, k_cache, v_cache, num_blocks, block_tables,
                       max_blocks_per_seq, context_lens, nullptr, nullptr, num_seqs, q_len,
                       num_q_heads, num_kv_heads, head_dim, block_size, 0, 1, nullptr, scale,
                       workspace, workspace_bytes, stream, k_scale, v_scale);
}

int pkv_paged_attn_decode_append(void* out, const void* q, const void* k_new, const void* v_new,
                                 void* k_cache, void* v_cache, int num_blocks,
                                 const int32_t* block_tables, int max_blocks_per_seq,
                                 const int32_t* context_lens, int num_seqs, int q_len,
                                 int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                 float scale, void* workspace, size_t workspace_bytes,
                                 pkv_stream_t stream) {
  if (num_seqs > 0 && (!k_new || !v_new)) return PKV_EINVAL;
  return launch_decode(false, out, q, num_seqs > 0 ? k_new : nullptr, v_new, k_cache, v_cache,
                       num_blocks, block_tables, max_blocks_per_seq, context_lens, nullptr,
                       nullptr, num_seqs, q_len, num_q_heads, num_kv_heads, head_dim, block_size,
                       0, 1, nullptr, scale, workspace, workspace_bytes, stream);
}

int pkv_ring_attn_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                         int num_blocks, const int32_t* block_tables, int max_blocks_per_seq,
                         const int64_t* logical_len, const int64_t* high_water, int num_seqs,
                         int q_len, int num_q_heads, int num_kv_heads, int head_dim,
                         int block_size, int sink, int window, const float* rope_cos_sin,
                         float scale, void* workspace, size_t workspace_bytes,
                         pkv_stream_t stream) {
  return launch_decode(true, out, q, nullptr, nullptr, k_cache, v_cache, num_blocks, block_tables,
                       max_blocks_per_seq, nullptr, logical_len, high_water, num_seqs, q_len,
                       num_q_heads, num_kv_heads, head_dim, block_size, sink, window,
                       rope_cos_sin, scale, workspace, workspace_bytes, stream);
}

int pkv_ring_attn_decode_append(void* out, const void* q, const void* k_new, const void* v_new,
                                void* k_cache, void* v_cache, int num_blocks,
                                const int32_t* block_tables, int max_blocks_per_seq,
                                const int64_t* logical_len, const int64_t* high_water,
                                int num_seqs, int q_len, int num_q_heads, int num_kv_heads,
                                int head_dim, int block_size, int sink, int window,
                                const float* rope_cos_sin, float scale, void* workspace,
                                size_t workspace_bytes, pkv_stream_t stream) {
  if (num_seqs > 0 && (!k_new || !v_new)) return PKV_EINVAL;
  return launch_decode(true, out, q, num_seqs > 0 ? k_new : nullptr, v_new, k_cache, v_cache,
                       num_blocks, block_tables, max_blocks_per_seq, nullptr, logical_len,
                       high_water, num_seqs, q_len, num_q_heads, num_kv_heads, head_dim,
                       block_size, sink, window, rope_cos_sin, scale, workspace, workspace_bytes,
                       stream);
}

int pkv_paged_attn_decode_noalloc(void* out, const void* q, const void* k_cache,
                                  const void* v_cache, int num_blocks,
                                  const int32_t* block_tables, int max_blocks_per_seq,
                                  const int32_t* context_lens, int num_seqs, int q_len,
                                  int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                  float scale, pkv_stream_t stream) {
  // the shape checks of pkv_paged_attn_decode, before anything else (an empty batch included)
  if (num_seqs < 0 || q_len < 1 || num_q_heads < 1 || num_kv_heads < 1 ||
      num_q_heads % num_kv_heads != 0 || head_dim != kD || !valid_block_size(block_size) ||
      num_blocks < 0 || max_blocks_per_seq < 0 || num_q_heads / num_kv_heads * q_len > 32)
    return PKV_EINVAL;
  if (num_seqs == 0) return PKV_OK;
  if (sm_count() == 0) return PKV_EINVAL;   // no usable current device
  const int R = num_q_heads / num_kv_heads * q_len;
  const WsLayout ws = ws_layout(num_seqs, num_kv_heads, R);
  if (ws.total > kFixedScratchBytes) return PKV_ENOSPC;
  int status = PKV_OK;
  void* scratch = fixed_scratch(&status);
  if (!scratch) return status;
  // the array keeps the previous call's contents; the arrival counters must start at zero
  const cudaError_t e = cudaMemsetAsync(scratch, 0, ws.part_ml, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_status(e);
  return pkv_paged_attn_decode(out, q, k_cache, v_cache, num_blocks, block_tables,
                               max_blocks_per_seq, context_lens, num_seqs, q_len, num_q_heads,
                               num_kv_heads, head_dim, block_size, scale, scratch,
                               kFixedScratchBytes, stream);
}

}  // extern "C"
