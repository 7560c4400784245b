// pkv_prefill.cu -- chunked-prefill paged attention on the 5th-generation tensor cores (sm_103a).
//
// What it computes ([VLLM] engineering trade-offs, chunked prefill: a long prompt is cut into
// chunks that go through attention over the paged cache): for sequence b, each of the chunk's
// q_len query tokens, at positions ctx - q_len + i, attends causally over the sequence's cached
// K/V (the chunk's own rows included, appended beforehand), read through the block table:
//   out[b][i][h] = softmax_t(scale * <q[b][i][h], K_t>) . V,   t < ctx - q_len + i + 1,
// the same operation as paged decode attention with a long query chunk.
//
// Design (GB300):
//  * Query tile = the G query heads of kv head h times TQ = 128 / G consecutive chunk tokens:
//    the 128 rows of one M = 128 MMA tile (row = token * G + head), so every K/V byte serves all
//    G heads. A CTA takes two query tiles of one (b, h) and every K/V stage it loads serves
//    both. CTAs of one (b, h) are launched next to each other (the longest tiles first), so
//    their shared K/V stays in L2.
//  * Keys in 64-token tiles: S = Q K^T (M 128, N 64, K 128) into tensor memory, then after the
//    softmax O += P V (M 128, N 128, K 64), with Q and P read from tensor memory (only K and V
//    come from shared memory, whose bandwidth the MMAs would otherwise saturate) and O
//    accumulated there for the whole context: tcgen05.mma kind::f16, f32 accumulate.
//  * Warp roles: warp 0 loads (TMA: the query tiles once, then K and V of each key tile as
//    16-token boxes at the rows the block table gives, into a 4-deep ring of 32 KB stages);
//    warp 1 allocates tensor memory (512 columns: S, O and Q of each tile) and issues the
//    MMAs, the whole warp running the issue loop and one elected lane issuing; warps 2-5 and
//    6-9 copy their query rows into tensor memory, then run the online softmax of tile 0 and
//    tile 1, one thread per row: S from tensor memory, mask, the row maximum by a tree, exp2
//    (the score scale folded into its argument), P (fp16) written back over S for the next
//    MMA.
//    The MMA order alternates the tiles (P_i(j) V_j, then S_i(j + 1)), so the tensor core works
//    on one tile while the other tile's softmax runs.
//  * The running maximum is raised only when a row's maximum grows by more than 2^8: the
//    factor e^(s - m) stays below 256 in fp16 and fp32, and O and the row sum are rescaled
//    (in tensor memory) only then; the result is the same up to rounding.
//  * Keys past those a tile needs are never read: boxes past them are out-of-range TMA loads
//    (zero fill). The last box loaded may reach past the context end; those rows are zeroed
//    in V before P V (they may hold anything, NaN included).
//  * Every wait is bounded: a wait that runs out sets PKV_DEVERR_TIMEOUT, the CTA winds down,
//    waits (bounded) for its copies and MMAs in flight and frees its tensor memory.
#include <cuda_fp16.h>

#include <algorithm>
#include <mutex>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kD = 128;
constexpr int kM = 128;              // rows of a query tile
constexpr int kKT = 64;              // keys per tile
#ifndef PKV_PREFILL_STAGES
#define PKV_PREFILL_STAGES 4
#endif
// Key tiles the loader warms L2 with ahead of the one it loads (0: none). A key tile is 16
// boxes from as many blocks; the first CTA of a (sequence, kv head) to need one misses L2.
#ifndef PKV_PREFILL_L2_AHEAD
#define PKV_PREFILL_L2_AHEAD 0
#endif
constexpr int kNS = PKV_PREFILL_STAGES;   // K/V stages
constexpr int kL2Ahead = PKV_PREFILL_L2_AHEAD;
constexpr int kThreads = 320;        // producer, MMA, 2 x 4 softmax warps
// S (and P over it) of tile i at 64 i; O of tile i at 128 + 128 i; Q of tile i at 384 + 64 i
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmO = 2 * 64, kTmQ = 2 * 64 + 2 * 128;
constexpr float kLazy = 8.0f;        // log2 of the largest factor before the max is raised
constexpr float kNegInf = -__builtin_huge_valf();
// A wait gives up after this long (a healthy pipeline waits microseconds).
constexpr uint64_t kWaitNs = 500ull * 1000 * 1000;

// shared memory (offsets from a 1024-byte aligned base)
constexpr int kQBytes = 2 * 16384;             // one query tile: lo / hi halves, 128 rows x 128 B
constexpr int kQ = 0;                          // two query tiles
constexpr int kStage0 = 2 * kQBytes;           // stages: K lo, K hi, V lo, V hi (64 rows x 128 B)
constexpr int kStageBytes = 4 * 8192;
constexpr int kBar = kStage0 + kNS * kStageBytes;
// barriers: kv_full[kNS], kv_empty[kNS], q_full, q_tmem, s_full[2], p_full[2], o_final
constexpr int kNumBars = 2 * kNS + 2 + 2 + 2 + 1;
constexpr int kMisc = kBar + kNumBars * 8;     // TMEM base address, abort flag
constexpr int kSmemBytes = kMisc + 16 + 1024;

struct PrefillArgs {
  __half* out;
  const int32_t* block_tables;
  const int32_t* context_lens;
  unsigned int* err;
  int num_blocks, max_blocks, num_seqs, q_len, Hq, Hkv, G, TQ, ntiles, npairs;
  int block_size, bs_shift;   // bs_shift = log2(block_size)
  float scale_log2;
};

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void flag_timeout(const PrefillArgs& a, volatile int* abort) {
  atomicOr(a.err, PKV_DEVERR_TIMEOUT);
  *abort = 1;
}

// Clamped context length of sequence b (sets PKV_DEVERR_CONTEXT when out of range).
__device__ __forceinline__ int context_of(const PrefillArgs& a, int b) {
  int ctx = __ldg(a.context_lens + b);
  const int lim = a.max_blocks * a.block_size;
  if (ctx < 0 || ctx > lim) ctx = ctx < 0 ? 0 : lim;
  return ctx;
}

// Keys query tile t needs: up to its last valid query's position (0 if the tile is past the
// chunk).
__device__ __forceinline__ int tile_kend(const PrefillArgs& a, int t, int ctx) {
  if (t >= a.ntiles) return 0;
  const int last_q = min(a.q_len, (t + 1) * a.TQ) - 1;
  return max(0, min(ctx, ctx - a.q_len + last_q + 1));
}

__global__ void __launch_bounds__(kThreads, 1)
prefill_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
               const __grid_constant__ CUtensorMap tmQ, const PrefillArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb0 = smem_u32(smem);
  const uint32_t bar_kv_full = sb0 + kBar;
  const uint32_t bar_kv_empty = bar_kv_full + kNS * 8;
  const uint32_t bar_q_full = bar_kv_empty + kNS * 8;
  const uint32_t bar_q_tmem = bar_q_full + 8;     // the queries are in tensor memory
  const uint32_t bar_s_full = bar_q_tmem + 8;     // [tile]
  const uint32_t bar_p_full = bar_s_full + 16;    // [tile]
  const uint32_t bar_o_final = bar_p_full + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kMisc);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + kMisc + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // unit: (b, h) groups in launch order, the pair of longest query tiles of a group first;
  // pair u holds query tiles 2 u and 2 u + 1
  const int grp = blockIdx.x / a.npairs;
  const int u = a.npairs - 1 - (blockIdx.x - grp * a.npairs);
  const int h = grp % a.Hkv, b = grp / a.Hkv;
  const int rows = a.TQ * a.G;              // rows of a tile in use
  const int raw_ctx = __ldg(a.context_lens + b);
  const int ctx = context_of(a, b);
  if (tid == 0 && raw_ctx != ctx) atomicOr(a.err, PKV_DEVERR_CONTEXT);
  const int first_pos = ctx - a.q_len;      // position of the chunk's first query
  const int t0 = 2 * u;
  const int kend0 = tile_kend(a, t0, ctx), kend1 = tile_kend(a, t0 + 1, ctx);
  const int nkt0 = (kend0 + kKT - 1) / kKT, nkt1 = (kend1 + kKT - 1) / kKT;
  const int kend = max(kend0, kend1);
  const int nkt = max(nkt0, nkt1);          // key tiles loaded (the later tile needs more)
  const int kpad = (kend + 15) & ~15;       // end of the last 16-token box loaded
  const bool has1 = t0 + 1 < a.ntiles;

  // ---- set-up: barriers, unused query rows zeroed, tensor memory -------------------------------
  if (tid == 0) {
    for (int s = 0; s < kNS; ++s) {
      mbar_init(bar_kv_full + s * 8, 1);
      mbar_init(bar_kv_empty + s * 8, 1);
    }
    mbar_init(bar_q_full, 1);
    mbar_init(bar_q_tmem, 256);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_s_full + i * 8, 1);
      mbar_init(bar_p_full + i * 8, 128);
    }
    mbar_init(bar_o_final, 1);
    *abort = 0;
  }
  // rows the query boxes do not cover still go through the MMA: make them finite (a missing
  // second tile is all zeros)
  for (int ti = 0; ti < 2; ++ti) {
    const int r0 = (ti == 0 || has1) ? rows : 0;
    for (int i = r0 * 8 + tid; i < kM * 8; i += kThreads) {
      reinterpret_cast<uint4*>(smem + kQ + ti * kQBytes)[i] = make_uint4(0, 0, 0, 0);
      reinterpret_cast<uint4*>(smem + kQ + ti * kQBytes + 16384)[i] = make_uint4(0, 0, 0, 0);
    }
  }
  fence_proxy_async_smem();
  fence_barrier_init();
  if (warp == 1) tmem_alloc(sb0 + kMisc, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // =================================== loads =================================================
    if (lane == 0) {
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
      prefetch_tensormap(&tmQ);
      mbar_arrive_expect_tx(bar_q_full, (has1 ? 2 : 1) * rows * 256);
      for (int ti = 0; ti < (has1 ? 2 : 1); ++ti) {
        const int qrow = b * a.q_len + (t0 + ti) * a.TQ;
        tma_load_3d(sb0 + kQ + ti * kQBytes, &tmQ, 0, h * a.G, qrow, bar_q_full);
        tma_load_3d(sb0 + kQ + ti * kQBytes + 16384, &tmQ, 64, h * a.G, qrow, bar_q_full);
      }
    }
    // K/V are read by every query tile of the unit: default L2 policy (they stay for the next)
    int issued = 0;
    // TMA row of box cc (< 4) of key tile jt, or -16 past the keys either query tile needs
    // (an out-of-range box: TMA fills it with zeros); `report` flags a bad block id
    auto box_row = [&](int jt, int cc, bool report) -> int {
      const int tok = jt * kKT + cc * 16;
      if (tok >= kend) return -16;
      const int blk = __ldg(a.block_tables + static_cast<int64_t>(b) * a.max_blocks +
                            (tok >> a.bs_shift));
      if (blk >= 0 && blk < a.num_blocks)
        return (blk * a.Hkv + h) * a.block_size + (tok & (a.block_size - 1));
      if (report) atomicOr(a.err, PKV_DEVERR_BLOCK_ID);
      return -16;
    };
    // warm L2 with the first key tiles (lanes: box lane / 4, part lane % 4)
    if (kL2Ahead > 0 && lane < 16) {
      for (int jt = 0; jt < min(nkt, kNS + kL2Ahead); ++jt) {
        const int r = box_row(jt, lane >> 2, false);
        if (r >= 0) tma_prefetch_l2_2d(((lane & 3) >> 1) ? &tmV : &tmK, (lane & 1) * 64, r);
      }
    }
    for (int j = 0; j < nkt; ++j) {
      if (__shfl_sync(0xffffffffu, *abort, 0)) break;    // one decision for the whole warp
      const int s = j % kNS;
      const int row = lane < 4 ? box_row(j, lane, true) : -16;
      // key tile j + kNS + kL2Ahead towards L2 while tile j's stage is awaited
      if (kL2Ahead > 0 && lane < 16 && j + kNS + kL2Ahead < nkt) {
        const int r = box_row(j + kNS + kL2Ahead, lane >> 2, false);
        if (r >= 0) tma_prefetch_l2_2d(((lane & 3) >> 1) ? &tmV : &tmK, (lane & 1) * 64, r);
      }
      if (lane == 0) {
        if (j >= kNS && !mbar_wait_ns(bar_kv_empty + s * 8, ((j / kNS) - 1) & 1, abort, kWaitNs))
          flag_timeout(a, abort);
        mbar_arrive_expect_tx(bar_kv_full + s * 8, kStageBytes);
      }
      __syncwarp();
      ++issued;
      // sixteen 2 KB boxes from sixteen lanes: box cc of K lo, K hi, V lo, V hi
      const int cc = lane >> 2, part = lane & 3;
      const int r = __shfl_sync(0xffffffffu, row, cc);
      if (lane < 16) {
        const uint32_t dst = sb0 + kStage0 + s * kStageBytes + (part >> 1) * 16384 +
                             (part & 1) * 8192 + cc * 2048;
        tma_load_2d(dst, (part >> 1) ? &tmV : &tmK, (part & 1) * 64, r, bar_kv_full + s * 8);
      }
    }
    // no TMA write may still be landing when the CTA leaves
    if (lane == 0) {
      for (int j = max(0, issued - kNS); j < issued; ++j)
        if (!mbar_wait_ns(bar_kv_full + (j % kNS) * 8, (j / kNS) & 1, nullptr, kWaitNs))
          flag_timeout(a, abort);
      if (!mbar_wait_ns(bar_q_full, 0, nullptr, kWaitNs)) flag_timeout(a, abort);
    }
    __syncwarp();
  } else if (warp == 1) {
    // =================================== MMA issue =============================================
    // Order: S_0(0), S_1(0); then per key tile j and query tile i: P_i(j) V_j, S_i(j + 1). A
    // commit tracks every MMA its thread issued before it, so when S_i(j + 1) is done
    // (s_full_i) P_i(j) V_j is too: the softmax of tile i may then overwrite P_i (written over
    // S_i) and rescale O_i. While one tile's softmax runs, the tensor core works on the other.
    // Q and P come from tensor memory: only K and V are read from shared memory.
    // The whole warp runs this loop (uniform control flow, every wait decided for the warp) and
    // one elected lane, the same every time, issues each MMA and commit: issued from a single
    // thread's branch, back-to-back MMAs with addresses computed in the loop went out at about
    // a third of the tensor core's rate.
    constexpr uint32_t idS = tc_idesc_f16(kM, kKT, false);
    constexpr uint32_t idO = tc_idesc_f16(kM, kD, true);
    const int nk[2] = {nkt0, has1 ? nkt1 : 0};
    auto wwait = [&](uint32_t bar, uint32_t parity, const volatile int* ab) -> bool {
      return __all_sync(0xffffffffu, mbar_wait_ns(bar, parity, ab, kWaitNs));
    };
    bool ok = nkt == 0 || wwait(bar_q_tmem, 0, abort);
    int waited = -1;                         // key tiles whose stage is known to have landed
    auto wait_kv = [&](int j) -> bool {
      while (waited < j) {
        const int jj = waited + 1;
        if (!wwait(bar_kv_full + (jj % kNS) * 8, (jj / kNS) & 1, abort)) return false;
        waited = jj;
      }
      return true;
    };
    auto issue_s = [&](int i, int j) {
      const uint32_t kst = sb0 + kStage0 + (j % kNS) * kStageBytes;
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t koff = (ks >> 2) * 8192 + (ks & 3) * 32;   // K lo/hi half
        // Q from tensor memory: 16 dims = 8 columns per step
        tc_mma_f16_ts_elect(tmem + i * kKT, tmem + kTmQ + i * kKT + ks * 8,
                            tc_desc_sw128(kst + koff, 16, 1024), idS, ks > 0);
      }
      tc_commit_elect(bar_s_full + i * 8);
    };
    for (int i = 0; ok && i < 2; ++i) {
      if (nk[i] == 0) continue;
      if (!(ok = wait_kv(0))) break;
      issue_s(i, 0);
    }
    for (int j = 0; ok && j < nkt; ++j) {
      for (int i = 0; i < 2; ++i) {
        if (j >= nk[i]) continue;
        if (!(ok = wwait(bar_p_full + i * 8, j & 1, abort))) break;
        tc_fence_after();
        const uint32_t vst = sb0 + kStage0 + (j % kNS) * kStageBytes + 16384;
#pragma unroll
        for (int kt = 0; kt < 4; ++kt) {
          // P from tensor memory (16 keys = 8 columns per step, over S_i); V: MN-major, 16
          // keys = two 8-row groups (1024 B apart), the dims' 64-column halves 8 KB apart
          tc_mma_f16_ts_elect(tmem + kTmO + i * kD, tmem + i * kKT + kt * 8,
                              tc_desc_sw128(vst + kt * 2048, 8192, 1024), idO,
                              (j > 0 || kt > 0));
        }
        if (j + 1 < nk[i]) {
          if (!(ok = wait_kv(j + 1))) break;
          issue_s(i, j + 1);
        }
      }
      if (!ok) break;
      // both tiles' P V of key tile j issued (a commit between them costs more than the stage
      // comes back earlier)
      tc_commit_elect(bar_kv_empty + (j % kNS) * 8);
    }
    if (!ok && lane == 0) flag_timeout(a, abort);
    // every MMA issued (all of them on the normal path) has completed when o_final fires
    tc_commit_elect(bar_o_final);
    if (!wwait(bar_o_final, 0, nullptr) && lane == 0) flag_timeout(a, abort);
  } else {
    // =================================== softmax ===============================================
    // Warps 2-5 take query tile 0, warps 6-9 tile 1, one thread per row. tcgen05.ld / st are
    // warp-collective (.sync.aligned): every decision that guards them (the waits, the rescale,
    // the epilogue) is taken for the whole warp.
    const int ti = (warp - 2) >> 2;             // query tile of this warp
    const int q4 = warp & 3;                    // TMEM lanes 32 q4 .. 32 q4 + 31
    const int r = 32 * q4 + lane;               // this thread's row
    const int tq = r / a.G, gh = r - tq * a.G;
    const int t = t0 + ti;
    const int qi = t * a.TQ + tq;
    const bool valid = t < a.ntiles && r < rows && qi < a.q_len;
    const int lim = valid ? max(0, min(ctx, first_pos + qi + 1)) : 0;   // keys t < lim visible
    const int my_nkt = ti == 0 ? nkt0 : (has1 ? nkt1 : 0);
    const uint32_t tl = tmem + (static_cast<uint32_t>(32 * q4) << 16);
    const uint32_t tO = tl + kTmO + ti * kD;
    const uint32_t tS = tl + ti * kKT;
    const int ptid = tid - 64 - ti * 128;       // 0 .. 127 within the softmax group
    auto warp_wait = [&](uint32_t bar, uint32_t parity) -> bool {
      const bool w = __all_sync(0xffffffffu, mbar_wait_ns(bar, parity, abort, kWaitNs));
      if (!w && lane == 0) flag_timeout(a, abort);
      return w;
    };
    const bool sl_pos = a.scale_log2 >= 0.f;
    float m_used = kNegInf, l = 0.f;
    bool ok = true;
    // this row of the query tile into tensor memory (the A operand of S = Q K^T): 128 dims,
    // two per column, from the 128-byte-swizzled lo / hi halves in shared memory
    if (nkt > 0) {                              // the MMA thread waits for all 256 rows
      ok = warp_wait(bar_q_full, 0);
      if (ok) {
        const uint32_t qt = sb0 + kQ + ti * kQBytes;
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t qr[32];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 v = ld_shared_v4(qt + hf * 16384 + r * 128 + ((c ^ (r & 7)) << 4));
            qr[4 * c] = v.x; qr[4 * c + 1] = v.y; qr[4 * c + 2] = v.z; qr[4 * c + 3] = v.w;
          }
          tmem_st32(tl + kTmQ + ti * kKT + hf * 32, qr);
        }
      }
      tc_fence_before();
      mbar_arrive(bar_q_tmem);
    }
    for (int j = 0; j < my_nkt; ++j) {
      // S_i(j) is done, and with it the P V of tile j - 1 (O is complete up to j - 1, P free)
      if (!(ok = warp_wait(bar_s_full + ti * 8, j & 1))) break;
      tc_fence_after();
      uint32_t sr[64];
      tmem_ld64(tS, sr);
      float x[64];
      const int base = j * kKT;
      float mx;
      const bool unmasked = base + kKT <= lim;
      if (unmasked) {
        // the scale is folded into the exponent below: the row's maximum of the raw scores
        // times the (positive) scale is the maximum of the scaled ones
#pragma unroll
        for (int i = 0; i < 64; ++i) x[i] = __uint_as_float(sr[i]);
        // a tree (8 chains of 8, then 3 levels): this reduction is on the tile's critical path
        // (the scale's sign, one decision for the launch, picks max or min outside the tree)
        float r8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) r8[k] = x[k];
        if (sl_pos) {
#pragma unroll
          for (int i = 8; i < 64; i += 8)
#pragma unroll
            for (int k = 0; k < 8; ++k) r8[k] = fmaxf(r8[k], x[i + k]);
#pragma unroll
          for (int w2 = 4; w2 >= 1; w2 >>= 1)
#pragma unroll
            for (int k = 0; k < w2; ++k) r8[k] = fmaxf(r8[k], r8[k + w2]);
        } else {
#pragma unroll
          for (int i = 8; i < 64; i += 8)
#pragma unroll
            for (int k = 0; k < 8; ++k) r8[k] = fminf(r8[k], x[i + k]);
#pragma unroll
          for (int w2 = 4; w2 >= 1; w2 >>= 1)
#pragma unroll
            for (int k = 0; k < w2; ++k) r8[k] = fminf(r8[k], r8[k + w2]);
        }
        mx = r8[0] * a.scale_log2;
      } else {
#pragma unroll
        for (int i = 0; i < 64; ++i)
          x[i] = base + i < lim ? __uint_as_float(sr[i]) * a.scale_log2 : kNegInf;
        float r8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) r8[k] = x[k];
#pragma unroll
        for (int i = 8; i < 64; i += 8)
#pragma unroll
          for (int k = 0; k < 8; ++k) r8[k] = fmaxf(r8[k], x[i + k]);
#pragma unroll
        for (int w2 = 4; w2 >= 1; w2 >>= 1)
#pragma unroll
          for (int k = 0; k < w2; ++k) r8[k] = fmaxf(r8[k], r8[k + w2]);
        mx = r8[0];
      }
      const bool raise = mx > m_used + kLazy;
      const bool resc = raise && m_used != kNegInf;   // this row's O and l need rescaling
      if (__any_sync(0xffffffffu, resc)) {
        // rescale the rows in place (factor 1 for the warp's other rows)
        const float f = resc ? fast_exp2(m_used - mx) : 1.f;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + 32 * c, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * f);
          tmem_st32(tO + 32 * c, o);
        }
        l *= f;
      }
      if (raise) m_used = mx;
      const float m_use = m_used == kNegInf ? 0.f : m_used;
      uint32_t ph[32];
      float rs[2] = {0.f, 0.f};                 // two partial sums: a shorter dependent chain
      if (unmasked) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float p0 = fast_exp2(fmaf(x[2 * i], a.scale_log2, -m_use));
          const float p1 = fast_exp2(fmaf(x[2 * i + 1], a.scale_log2, -m_use));
          rs[i & 1] += p0 + p1;
          ph[i] = pack_half2(p0, p1);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float p0 = fast_exp2(x[2 * i] - m_use), p1 = fast_exp2(x[2 * i + 1] - m_use);
          rs[i & 1] += p0 + p1;
          ph[i] = pack_half2(p0, p1);
        }
      }
      l += rs[0] + rs[1];
      // the last box loaded ends at kpad; its rows at or past the context end may hold
      // anything: zero them in V before P V reads them (P is 0 there, but 0 x NaN is not).
      // Both groups zero the same rows when both use the tile (the same bytes).
      const int s = j % kNS;
      if (j == nkt - 1 && kpad > ctx) {
        if (!(ok = warp_wait(bar_kv_full + s * 8, (j / kNS) & 1))) break;
        const int r0 = ctx - base, r1 = kpad - base;
        const int n = (r1 - r0) * 16;             // 16-byte pieces: rows x (2 halves x 8)
        for (int i = ptid; i < n; i += 128) {
          const int rr = r0 + i / 16, piece = i % 16;
          const uint32_t addr = sb0 + kStage0 + s * kStageBytes + 16384 + (piece >> 3) * 8192 +
                                rr * 128 + (piece & 7) * 16;
          st_shared_v4(addr, make_uint4(0, 0, 0, 0));
        }
        fence_proxy_async_smem();
      }
      // P (fp16, two per column) over the first 32 columns of the tile's S, read by P V
      tmem_st32(tS, ph);
      tc_fence_before();
      mbar_arrive(bar_p_full + ti * 8);
    }
    // ---- epilogue: O / l, fp16, to the output row ----------------------------------------------
    const bool have_o = ok && my_nkt > 0 && warp_wait(bar_o_final, 0);
    const float inv = (have_o && l > 0.f) ? 1.f / l : 0.f;
    __half* dst = a.out + ((static_cast<int64_t>(b) * a.q_len + qi) * a.Hq + h * a.G + gh) * kD;
    if (have_o) tc_fence_after();
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      uint32_t o[32];
      if (have_o) {
        tmem_ld32(tO + 32 * c, o);              // the whole warp, valid rows or not
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = 0u;
      }
      if (valid) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint4 v;
          v.x = pack_half2(__uint_as_float(o[8 * i + 0]) * inv, __uint_as_float(o[8 * i + 1]) * inv);
          v.y = pack_half2(__uint_as_float(o[8 * i + 2]) * inv, __uint_as_float(o[8 * i + 3]) * inv);
          v.z = pack_half2(__uint_as_float(o[8 * i + 4]) * inv, __uint_as_float(o[8 * i + 5]) * inv);
          v.w = pack_half2(__uint_as_float(o[8 * i + 6]) * inv, __uint_as_float(o[8 * i + 7]) * inv);
          *reinterpret_cast<uint4*>(dst + 32 * c + 8 * i) = v;
        }
      }
    }
    tc_fence_before();
  }
  // ---- teardown: every copy and MMA of this CTA has landed; free the tensor memory -------------
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

int encode(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims,
           const cuuint64_t* strides, const cuuint32_t* box) {
  auto fn = tensor_map_encoder();
  if (!fn) return PKV_ECUDA_BASE - static_cast<int>(cudaErrorNotSupported);
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, rank, const_cast<void*>(base), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PKV_OK : PKV_EINVAL;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" int pkv_paged_prefill(void* out, const void* q, const void* k_cache,
                                 const void* v_cache, int num_blocks,
                                 const int32_t* block_tables, int max_blocks_per_seq,
                                 const int32_t* context_lens, int num_seqs, int q_len,
                                 int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                 float scale, pkv_stream_t stream) {
  if (num_seqs < 0 || q_len < 1 || num_q_heads < 1 || num_kv_heads < 1 ||
      num_q_heads % num_kv_heads != 0 || head_dim != kD || !valid_block_size(block_size) ||
      num_blocks < 1 || max_blocks_per_seq < 0)
    return PKV_EINVAL;
  const int G = num_q_heads / num_kv_heads;
  if (G > kM) return PKV_EINVAL;
  if (num_seqs == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens) return PKV_EINVAL;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return PKV_EINVAL;
  const int64_t rows = static_cast<int64_t>(num_blocks) * num_kv_heads * block_size;
  const int64_t qrows = static_cast<int64_t>(num_seqs) * q_len;
  // query tokens per tile: as many as fill the 128 rows, at most the chunk (so that the query
  // box never exceeds the query tensor)
  const int TQ = std::min(kM / G, q_len);
  const int64_t ntiles = (q_len + TQ - 1) / TQ;
  const int64_t npairs = (ntiles + 1) / 2;        // two query tiles per CTA
  const int64_t grid = npairs * num_kv_heads * num_seqs;
  if (rows >= (1ll << 31) || qrows >= (1ll << 31) || grid >= (1ll << 31) ||
      static_cast<int64_t>(max_blocks_per_seq) * block_size >= (1ll << 30))
    return PKV_EINVAL;

  {
    // the shared-memory limit is a per-device attribute of the kernel: raise it once per device
    static std::mutex mu;
    static bool done[64] = {};
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_status(e);
    if (dev < 0 || dev >= 64) return PKV_EINVAL;
    std::lock_guard<std::mutex> lock(mu);
    if (!done[dev]) {
      e = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kSmemBytes);
      if (e != cudaSuccess) return cuda_status(e);
      done[dev] = true;
    }
  }

  CUtensorMap tmK, tmV, tmQ;
  const cuuint64_t kv_dims[2] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(rows)};
  const cuuint64_t kv_strides[1] = {kD * 2};
  const cuuint32_t kv_box[2] = {64, 16};
  int st = encode(&tmK, k_cache, 2, kv_dims, kv_strides, kv_box);
  if (st == PKV_OK) st = encode(&tmV, v_cache, 2, kv_dims, kv_strides, kv_box);
  const cuuint64_t q_dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(num_q_heads),
                                static_cast<cuuint64_t>(qrows)};
  const cuuint64_t q_strides[2] = {kD * 2, static_cast<cuuint64_t>(num_q_heads) * kD * 2};
  const cuuint32_t q_box[3] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(TQ)};
  if (st == PKV_OK) st = encode(&tmQ, q, 3, q_dims, q_strides, q_box);
  if (st != PKV_OK) return st;

  unsigned int* err = device_error_ptr();
  if (!err) return PKV_EINVAL;
  PrefillArgs args;
  args.out = static_cast<__half*>(out);
  args.block_tables = block_tables;
  args.context_lens = context_lens;
  args.err = err;
  args.num_blocks = num_blocks;
  args.max_blocks = max_blocks_per_seq;
  args.num_seqs = num_seqs;
  args.q_len = q_len;
  args.Hq = num_q_heads;
  args.Hkv = num_kv_heads;
  args.G = G;
  args.TQ = TQ;
  args.ntiles = static_cast<int>(ntiles);
  args.npairs = static_cast<int>(npairs);
  args.block_size = block_size;
  int shift = 0;
  while ((1 << shift) < block_size) ++shift;
  args.bs_shift = shift;
  args.scale_log2 = scale * 1.4426950408889634f;
  prefill_kernel<<<static_cast<unsigned>(grid), kThreads, kSmemBytes,
                   static_cast<cudaStream_t>(stream)>>>(tmK, tmV, tmQ, args);
  return cuda_status(cudaGetLastError());
}
