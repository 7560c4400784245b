// pkv_oracle.cpp -- TEST INFRASTRUCTURE ONLY.
//
// A plain, slow, fp64 CPU statement of what paged KV-cache decode attention
// computes. It exists so that the CUDA library can be checked against it;
// nothing in the product may link, load or call it. Only the test suite,
// the smoke check and the benchmark's CPU-baseline leg use it.
//
// It shares no code, header, table or constant generator with the CUDA path.
// Every function restates a passage of the source pages; the citation names
// the page and the section. Pages:
//   [EDGE]   "端侧 SLM 显存保活术：在 4GB 内存板卡上实现轻量 PagedAttention 与
//             KV 缓存分块" (sheratonhq.com/news/141880)
//   [OLLAMA] "Ollama的内存管理策略：从KV Cache Block分配到Prefix-aware内存复用
//             的演进" (xdnf.cn/news/5086)
//   [RING]   streaming-inference page on deferred speculative decoding and
//             circular context (wzjinhao.cn/news/69573)
//   [VLLM]   "大模型推理内存优化：从 KV Cache 分页到连续批处理的工程实践"
//             (pwwt.cn/news/3010209)
//
// Conventions fixed here (the pages are silent on them, so each is a reading of
// them, chosen as the plainest one the rest of the pages support):
//   * KV pool of one layer: [num_blocks][num_kv_heads][block_size][head_dim],
//     fp16 stored as raw uint16 bit patterns, K and V in separate pools.
//   * GQA: query head h reads kv head h / (num_q_heads / num_kv_heads).
//   * context_lens counts the tokens in cache after this step's append.
//   * With q_len > 1 the queries are the last q_len tokens of the sequence and
//     query i sees tokens [0, ctx - q_len + i + 1) (causal).
//   * A negative slot in a slot mapping is padding and is skipped.
//
// Parity status: every function here is pinned by the CPU tests against the
// pages' printed numbers, closed forms, library routines or brute force,
// except the ring valid-set rule after a rollback (pkv_orc_ring_valid), whose
// reading is pinned only by an independent linear-history simulation: the
// pages do not fix it ("parity unpinned" against the pages for that rule).

#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>
#include <algorithm>

namespace {

// ---------------------------------------------------------------------------
// Textbook attention of one query vector over an explicit list of keys:
// s_t = scale * <q, K_t>, p = softmax(s), out = sum_t p_t V_t. fp64 throughout.
// ---------------------------------------------------------------------------
static void attend(const double* q, const std::vector<double>& K, const std::vector<double>& V,
                   int64_t n, int D, double scale, double* out) {
  if (n == 0) { for (int d = 0; d < D; ++d) out[d] = 0.0; return; }
  std::vector<double> s(n);
  double m = -INFINITY;
  for (int64_t t = 0; t < n; ++t) {
    double acc = 0.0;
    for (int d = 0; d < D; ++d) acc += q[d] * K[t * D + d];
    s[t] = scale * acc;
    m = std::max(m, s[t]);
  }
  double l = 0.0;
  for (int64_t t = 0; t < n; ++t) { s[t] = std::exp(s[t] - m); l += s[t]; }
  for (int d = 0; d < D; ++d) {
    double acc = 0.0;
    for (int64_t t = 0; t < n; ++t) acc += s[t] * V[t * D + d];
    out[d] = acc / l;
  }
}

// Runs fn(item) for item in [0, n_items) on num_threads threads (0 = all cores).
template <class F>
static int parallel_for(int64_t n_items, int num_threads, F fn) {
  int nt = num_threads > 0 ? num_threads : static_cast<int>(std::thread::hardware_concurrency());
  if (nt < 1) nt = 1;
  if (nt > n_items) nt = static_cast<int>(std::max<int64_t>(1, n_items));
  std::vector<std::thread> pool;
  for (int w = 0; w < nt; ++w)
    pool.emplace_back([=]() { for (int64_t i = w; i < n_items; i += nt) fn(i); });
  for (auto& th : pool) th.join();
  return nt;
}

}  // namespace

extern "C" {

// ---------------------------------------------------------------------------
// KV byte ledger.
// [VLLM] §KV Cache 的内存开销与分页机制: KV size = 2 x layers x seq_len x
// kv_heads x head_dim x dtype_size x batch. [EDGE] §KV Cache 的物理膨胀账本
// gives the per-layer, per-token form (2 x kv_heads x head_dim x 2 bytes).
// ---------------------------------------------------------------------------
uint64_t pkv_orc_kv_bytes(uint64_t num_layers, uint64_t seq_len, uint64_t num_kv_heads,
                          uint64_t head_dim, uint64_t dtype_bytes, uint64_t batch) {
  return 2ull * num_layers * seq_len * num_kv_heads * head_dim * dtype_bytes * batch;
}

// ---------------------------------------------------------------------------
// IEEE-754 binary16 -> binary64, from the format's definition (1 sign bit,
// 5 exponent bits with bias 15, 10 fraction bits; exponent 0 = subnormal,
// exponent 31 = inf/NaN). Exact: every binary16 value is a binary64 value.
// ---------------------------------------------------------------------------
double pkv_orc_f16_to_f64(uint16_t h) {
  const int sign = (h >> 15) & 1;
  const int expo = (h >> 10) & 0x1f;
  const int frac = h & 0x3ff;
  double v;
  if (expo == 0) {
    v = std::ldexp(static_cast<double>(frac), -24);            // frac * 2^-14 * 2^-10
  } else if (expo == 31) {
    v = frac ? std::nan("") : INFINITY;
  } else {
    v = std::ldexp(static_cast<double>(frac | 0x400), expo - 25);  // 1.frac * 2^(e-15)
  }
  return sign ? -v : v;
}

void pkv_orc_f16_array_to_f64(const uint16_t* src, double* dst, int64_t n) {
  for (int64_t i = 0; i < n; ++i) dst[i] = pkv_orc_f16_to_f64(src[i]);
}

// ---------------------------------------------------------------------------
// Paged slot mapping.
// [EDGE] §注意力寻址非连续物理块的间接寻址内核: logical block = T / TOKENS_PER_BLOCK,
// offset = T % TOKENS_PER_BLOCK, physical block = block_table[logical block].
// [VLLM] (paging list, 按需分配): a new token goes into the sequence's current
// block. A slot is physical_block * block_size + offset. A negative position
// gives slot -1 (padding).
// ---------------------------------------------------------------------------
void pkv_orc_slot_mapping(const int32_t* seq_ids, const int64_t* positions, int n,
                          const int32_t* block_tables, int max_blocks_per_seq,
                          int block_size, int64_t* slot_out) {
  for (int i = 0; i < n; ++i) {
    const int64_t p = positions[i];
    if (p < 0) { slot_out[i] = -1; continue; }
    const int64_t logical_block = p / block_size;
    const int64_t offset = p % block_size;
    const int64_t phys =
        block_tables[static_cast<int64_t>(seq_ids[i]) * max_blocks_per_seq + logical_block];
    slot_out[i] = phys * block_size + offset;
  }
}

// ---------------------------------------------------------------------------
// Sink + ring slot.
// [RING] §环形上下文与注意力沉淀机制: Slot(pos) = pos for pos < S, and
// S + ((pos - S) mod W) for pos >= S.
// ---------------------------------------------------------------------------
int64_t pkv_orc_ring_slot(int64_t pos, int64_t sink, int64_t window) {
  if (pos < sink) return pos;
  return sink + (pos - sink) % window;
}

// Ring slot r lives in the paged pool at block_table[b][r / bs], offset r % bs.
void pkv_orc_ring_slot_mapping(const int32_t* seq_ids, const int64_t* positions, int n,
                               const int32_t* block_tables, int max_blocks_per_seq,
                               int sink, int window, int block_size, int64_t* slot_out) {
  for (int i = 0; i < n; ++i) {
    const int64_t p = positions[i];
    if (p < 0) { slot_out[i] = -1; continue; }
    const int64_t r = pkv_orc_ring_slot(p, sink, window);
    const int64_t phys =
        block_tables[static_cast<int64_t>(seq_ids[i]) * max_blocks_per_seq + r / block_size];
    slot_out[i] = phys * block_size + r % block_size;
  }
}

// Valid logical positions seen by query qi of a ring sequence, in logical
// order. [RING] §C 环形 KV 缓存管理内核实现 (FillValidPhysicalIndices) lists the
// sinks followed by the last W positions. Reading kept here: with a
// high-water mark hw (one past the largest position ever written) the window
// part is [max(S, hw - W), vis) where vis = L - q_len + qi + 1 is the causal
// limit of query qi; with hw == L and q_len == 1 this is the page's list.
// Precondition: hw - W <= L <= hw (a rollback never goes deeper than the
// window), under which the positions [max(S, hw - W), hw) are exactly the
// ones still physically present in the window slots.
// Returns the count; positions go to out (capacity >= S + W).
int pkv_orc_ring_valid(int64_t L, int64_t hw, int sink, int window, int q_len, int qi,
                       int64_t* out) {
  const int64_t vis = L - q_len + qi + 1;
  int n = 0;
  for (int64_t p = 0; p < sink && p < vis; ++p) out[n++] = p;
  const int64_t lo = std::max<int64_t>(sink, hw - window);
  for (int64_t p = lo; p < vis; ++p) out[n++] = p;
  return n;
}

// ---------------------------------------------------------------------------
// KV append: [VLLM] paging list (按需分配) and [RING] AppendKV: the new token's
// K/V vectors are copied into its slot. Byte copy; slot < 0 is skipped.
// k, v: [num_tokens][num_kv_heads][head_dim]; caches: one layer.
// ---------------------------------------------------------------------------
void pkv_orc_kv_append(const uint16_t* k, const uint16_t* v, const int64_t* slot_mapping,
                       int num_tokens, uint16_t* k_cache, uint16_t* v_cache,
                       int num_kv_heads, int head_dim, int block_size) {
  for (int t = 0; t < num_tokens; ++t) {
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    const int64_t blk = slot / block_size, off = slot % block_size;
    for (int h = 0; h < num_kv_heads; ++h) {
      const int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * head_dim;
      const int64_t src = (static_cast<int64_t>(t) * num_kv_heads + h) * head_dim;
      std::memcpy(k_cache + dst, k + src, sizeof(uint16_t) * head_dim);
      std::memcpy(v_cache + dst, v + src, sizeof(uint16_t) * head_dim);
    }
  }
}

// ---------------------------------------------------------------------------
// Copy-on-write block copy. [OLLAMA] §三 (CoW paragraph): a writer to a shared,
// reference-counted block first copies the block and writes to the copy.
// Copies block src[i] -> dst[i] in every layer, K and V.
// ---------------------------------------------------------------------------
void pkv_orc_copy_blocks(uint16_t* k_cache, uint16_t* v_cache, const int32_t* src,
                         const int32_t* dst, int n, int64_t layer_stride_elems,
                         int num_layers, int64_t block_elems) {
  for (int l = 0; l < num_layers; ++l) {
    for (int i = 0; i < n; ++i) {
      const int64_t s = l * layer_stride_elems + static_cast<int64_t>(src[i]) * block_elems;
      const int64_t d = l * layer_stride_elems + static_cast<int64_t>(dst[i]) * block_elems;
      std::memmove(k_cache + d, k_cache + s, sizeof(uint16_t) * block_elems);
      std::memmove(v_cache + d, v_cache + s, sizeof(uint16_t) * block_elems);
    }
  }
}

// ---------------------------------------------------------------------------
// Paged decode attention (the method's result, written as its definition).
// [EDGE] §注意力寻址非连续物理块的间接寻址内核 (addressing) and [VLLM] paging list
// and PagedAttention-kernel paragraph (the kernel reads K/V indirectly through
// the block table): gather each sequence's K/V rows in logical order through
// its block table, converting fp16 -> fp64, then run textbook softmax
// attention over them.
//   q:   [B][q_len][Hq][D] fp16     out: [B][q_len][Hq][D] fp64
//   block_tables: [B][max_blocks_per_seq]; context_lens: [B]
//   seq_mask: optional [B] bytes; sequences with 0 are skipped (out untouched).
// Returns the number of threads used.
// ---------------------------------------------------------------------------
int pkv_orc_paged_attention(double* out, const uint16_t* q, const uint16_t* k_cache,
                            const uint16_t* v_cache, const int32_t* block_tables,
                            int max_blocks_per_seq, const int32_t* context_lens, int B,
                            int q_len, int Hq, int Hkv, int D, int block_size, double scale,
                            const uint8_t* seq_mask, int num_threads) {
  const int G = Hq / Hkv;
  const int64_t items = static_cast<int64_t>(B) * Hkv;
  return parallel_for(items, num_threads, [&](int64_t item) {
    const int b = static_cast<int>(item / Hkv), kvh = static_cast<int>(item % Hkv);
    if (seq_mask && !seq_mask[b]) return;
    const int64_t ctx = context_lens[b];
    // Gather this (sequence, kv head)'s keys and values in logical order.
    std::vector<double> K(ctx * D), V(ctx * D);
    for (int64_t t = 0; t < ctx; ++t) {
      const int64_t phys = block_tables[static_cast<int64_t>(b) * max_blocks_per_seq + t / block_size];
      const int64_t row = ((phys * Hkv + kvh) * block_size + t % block_size) * D;
      for (int d = 0; d < D; ++d) {
        K[t * D + d] = pkv_orc_f16_to_f64(k_cache[row + d]);
        V[t * D + d] = pkv_orc_f16_to_f64(v_cache[row + d]);
      }
    }
    std::vector<double> qv(D);
    for (int qi = 0; qi < q_len; ++qi) {
      const int64_t visible = std::max<int64_t>(0, ctx - q_len + qi + 1);
      for (int g = 0; g < G; ++g) {
        const int h = kvh * G + g;
        const int64_t base = ((static_cast<int64_t>(b) * q_len + qi) * Hq + h) * D;
        for (int d = 0; d < D; ++d) qv[d] = pkv_orc_f16_to_f64(q[base + d]);
        attend(qv.data(), K, V, visible, D, scale, out + base);
      }
    }
  });
}

// ---------------------------------------------------------------------------
// Rotary position embedding, rotate-half form, fp64.
// [RING] §环形上下文与注意力沉淀机制: as the ring wraps, historic keys are rotated
// so that the query-key dot product keeps the right relative distance. The
// rotation: pairs (i, i + D/2), theta_i = base^(-2i/D), angle = index * theta_i.
// ---------------------------------------------------------------------------
void pkv_orc_rope(double* x, int D, double index, double base) {
  const int half = D / 2;
  for (int i = 0; i < half; ++i) {
    const double theta = std::pow(base, -2.0 * i / D);
    const double c = std::cos(index * theta), s = std::sin(index * theta);
    const double a = x[i], b = x[i + half];
    x[i] = a * c - b * s;
    x[i + half] = b * c + a * s;
  }
}

// ---------------------------------------------------------------------------
// Sink + ring decode attention. [RING] §环形上下文与注意力沉淀机制 and
// §C 环形 KV 缓存管理内核实现. Position p of sequence b is stored at ring slot
// Slot(p), which lives in the paged pool through block_table[b]. Query qi
// (position L - q_len + qi) sees the positions listed by pkv_orc_ring_valid.
// Keys are stored before RoPE; rope_mode chooses the rotation index:
//   0: cache index (sinks 0..S-1, then the window oldest -> newest numbered
//      from S), the query using its own key's cache index;
//   1: true logical position for both;  2: no rotation.
// logical_len[b] = L (after this step's appends); high_water[b] = hw.
// ---------------------------------------------------------------------------
int pkv_orc_ring_attention(double* out, const uint16_t* q, const uint16_t* k_cache,
                           const uint16_t* v_cache, const int32_t* block_tables,
                           int max_blocks_per_seq, const int64_t* logical_len,
                           const int64_t* high_water, int B, int q_len, int Hq, int Hkv,
                           int D, int block_size, int sink, int window, double scale,
                           int rope_mode, double rope_base, const uint8_t* seq_mask,
                           int num_threads) {
  const int G = Hq / Hkv;
  const int64_t items = static_cast<int64_t>(B) * Hkv;
  return parallel_for(items, num_threads, [&](int64_t item) {
    const int b = static_cast<int>(item / Hkv), kvh = static_cast<int>(item % Hkv);
    if (seq_mask && !seq_mask[b]) return;
    const int64_t L = logical_len[b], hw = high_water[b];
    const int64_t lo = std::max<int64_t>(sink, hw - window);
    auto cache_index = [&](int64_t p) -> double {
      if (rope_mode == 1) return static_cast<double>(p);
      return static_cast<double>(p < sink ? p : sink + (p - lo));
    };
    std::vector<int64_t> pos(sink + window + 1);
    std::vector<double> qv(D);
    for (int qi = 0; qi < q_len; ++qi) {
      const int n = pkv_orc_ring_valid(L, hw, sink, window, q_len, qi, pos.data());
      std::vector<double> K(static_cast<int64_t>(n) * D), V(static_cast<int64_t>(n) * D);
      for (int t = 0; t < n; ++t) {
        const int64_t r = pkv_orc_ring_slot(pos[t], sink, window);
        const int64_t phys = block_tables[static_cast<int64_t>(b) * max_blocks_per_seq + r / block_size];
        const int64_t row = ((phys * Hkv + kvh) * block_size + r % block_size) * D;
        for (int d = 0; d < D; ++d) {
          K[static_cast<int64_t>(t) * D + d] = pkv_orc_f16_to_f64(k_cache[row + d]);
          V[static_cast<int64_t>(t) * D + d] = pkv_orc_f16_to_f64(v_cache[row + d]);
        }
        if (rope_mode != 2) pkv_orc_rope(&K[static_cast<int64_t>(t) * D], D, cache_index(pos[t]), rope_base);
      }
      const int64_t qpos = L - q_len + qi;
      for (int g = 0; g < G; ++g) {
        const int h = kvh * G + g;
        const int64_t base = ((static_cast<int64_t>(b) * q_len + qi) * Hq + h) * D;
        for (int d = 0; d < D; ++d) qv[d] = pkv_orc_f16_to_f64(q[base + d]);
        if (rope_mode != 2) pkv_orc_rope(qv.data(), D, cache_index(qpos), rope_base);
        attend(qv.data(), K, V, n, D, scale, out + base);
      }
    }
  });
}


// ---------------------------------------------------------------------------
// FP8 KV cache (E4M3).
// [VLLM] §工程权衡 (量化与 KV Cache 精度的权衡): quantising the KV cache from FP16
// to FP8 halves its memory, and production keeps KV at FP8 rather than INT4.
// The page names no FP8 layout; the reading here is the E4M3 format (1 sign
// bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent 0 subnormal;
// S.1111.111 is NaN and there is no infinity, so the largest finite value is
// 1.75 * 2^8 = 448), one scale per (layer, kv head) for K and one for V:
// stored code = E4M3(x / scale), value = decode(code) * scale.
// ---------------------------------------------------------------------------
double pkv_orc_e4m3_to_f64(uint8_t c) {
  const int sign = (c >> 7) & 1;
  const int expo = (c >> 3) & 0xf;
  const int mant = c & 7;
  double v;
  if (expo == 15 && mant == 7) return std::nan("");
  if (expo == 0)
    v = std::ldexp(static_cast<double>(mant), -9);             // mant/8 * 2^-6
  else
    v = std::ldexp(static_cast<double>(8 + mant), expo - 10);  // (1 + mant/8) * 2^(e-7)
  return sign ? -v : v;
}

// Round to the nearest E4M3 value, ties to the even code (mantissa bit 0 clear), finite
// values beyond the largest saturate to +-448, NaN stays NaN. Plain search over the codes.
uint8_t pkv_orc_f64_to_e4m3(double x) {
  const uint8_t sign = std::signbit(x) ? 0x80 : 0x00;
  if (std::isnan(x)) return sign | 0x7f;
  const double a = std::fabs(x);
  if (a >= 448.0) return sign | 0x7e;
  int best = 0;
  double best_err = INFINITY;
  for (int c = 0; c <= 0x7e; ++c) {
    const double err = std::fabs(pkv_orc_e4m3_to_f64(static_cast<uint8_t>(c)) - a);
    if (err < best_err || (err == best_err && (c & 1) == 0)) { best = c; best_err = err; }
  }
  return sign | static_cast<uint8_t>(best);
}

// FP8 append: the FP16 row's elements, divided by their kv head's scale in
// binary32 (the precision the device takes the quantisation decision in), go
// to E4M3 codes in the pools' slots. Pools: [NB][Hkv][bs][D] bytes.
void pkv_orc_kv_append_fp8(const uint16_t* k, const uint16_t* v, const int64_t* slot_mapping,
                           int num_tokens, uint8_t* k_cache, uint8_t* v_cache,
                           int num_kv_heads, int D, int block_size, const float* k_scale,
                           const float* v_scale) {
  for (int t = 0; t < num_tokens; ++t) {
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    const int64_t blk = slot / block_size, off = slot % block_size;
    for (int h = 0; h < num_kv_heads; ++h) {
      const int64_t src = (static_cast<int64_t>(t) * num_kv_heads + h) * D;
      const int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * D;
      for (int d = 0; d < D; ++d) {
        const float xk = static_cast<float>(pkv_orc_f16_to_f64(k[src + d])) / k_scale[h];
        const float xv = static_cast<float>(pkv_orc_f16_to_f64(v[src + d])) / v_scale[h];
        k_cache[dst + d] = pkv_orc_f64_to_e4m3(xk);
        v_cache[dst + d] = pkv_orc_f64_to_e4m3(xv);
      }
    }
  }
}

// Paged decode attention over an FP8 cache: the same gather-then-textbook
// attention as pkv_orc_paged_attention, each K (V) element being
// decode(code) * k_scale[kv head] (v_scale) in fp64.
int pkv_orc_paged_attention_fp8(double* out, const uint16_t* q, const uint8_t* k_cache,
                                const uint8_t* v_cache, const float* k_scale,
                                const float* v_scale, const int32_t* block_tables,
                                int max_blocks_per_seq, const int32_t* context_lens, int B,
                                int q_len, int Hq, int Hkv, int D, int block_size, double scale,
                                int num_threads) {
  const int G = Hq / Hkv;
  const int64_t items = static_cast<int64_t>(B) * Hkv;
  return parallel_for(items, num_threads, [&](int64_t item) {
    const int b = static_cast<int>(item / Hkv), kvh = static_cast<int>(item % Hkv);
    const int64_t ctx = context_lens[b];
    std::vector<double> K(ctx * D), V(ctx * D);
    for (int64_t t = 0; t < ctx; ++t) {
      const int64_t phys = block_tables[static_cast<int64_t>(b) * max_blocks_per_seq + t / block_size];
      const int64_t row = ((phys * Hkv + kvh) * block_size + t % block_size) * D;
      for (int d = 0; d < D; ++d) {
        K[t * D + d] = pkv_orc_e4m3_to_f64(k_cache[row + d]) * static_cast<double>(k_scale[kvh]);
        V[t * D + d] = pkv_orc_e4m3_to_f64(v_cache[row + d]) * static_cast<double>(v_scale[kvh]);
      }
    }
    std::vector<double> qv(D);
    for (int qi = 0; qi < q_len; ++qi) {
      const int64_t visible = std::max<int64_t>(0, ctx - q_len + qi + 1);
      for (int g = 0; g < G; ++g) {
        const int h = kvh * G + g;
        const int64_t base = ((static_cast<int64_t>(b) * q_len + qi) * Hq + h) * D;
        for (int d = 0; d < D; ++d) qv[d] = pkv_orc_f16_to_f64(q[base + d]);
        attend(qv.data(), K, V, visible, D, scale, out + base);
      }
    }
  });
}


// ---------------------------------------------------------------------------
// Speculative verification of K draft tokens per sequence.
// [RING] (deferred speculative decoding paragraph): the target model accepts
// draft token x with probability min(1, P_target(x) / P_draft(x)); the first
// rejection ends the accepted run (the rejected drafts are rolled back).
// Readings (the page leaves them to the standard method): the draws are
// given, u_accept[b][k] in [0, 1) per draft and u_sample[b] per sequence;
// draft k is accepted iff u_accept * P_draft(x) < P_target(x); after a
// rejection at k the next token is drawn from the normalised residual
// max(0, P_target - P_draft) at k, after K acceptances from P_target at
// position K, by inverse CDF: the first v whose cumulative weight exceeds
// u_sample times the total. P = softmax of the given logits, fp64 here.
//   target_logits [B][K+1][V], draft_logits [B][K][V], drafts [B][K]
// ---------------------------------------------------------------------------
void pkv_orc_spec_verify(const float* target_logits, const float* draft_logits,
                         const int32_t* drafts, const float* u_accept, const float* u_sample,
                         int B, int K, int V, int32_t* n_accept, int32_t* next_token) {
  auto softmax = [V](const float* x, std::vector<double>& p) {
    double m = -INFINITY;
    for (int v = 0; v < V; ++v) m = std::max(m, static_cast<double>(x[v]));
    double s = 0.0;
    for (int v = 0; v < V; ++v) { p[v] = std::exp(static_cast<double>(x[v]) - m); s += p[v]; }
    for (int v = 0; v < V; ++v) p[v] /= s;
  };
  auto draw = [V](const std::vector<double>& w, double u) {
    double total = 0.0;
    for (int v = 0; v < V; ++v) total += w[v];
    const double thr = u * total;
    double c = 0.0;
    for (int v = 0; v < V; ++v) {
      c += w[v];
      if (c > thr) return v;
    }
    return V - 1;
  };
  std::vector<double> pt(V), pd(V), r(V);
  for (int b = 0; b < B; ++b) {
    int k = 0;
    for (; k < K; ++k) {
      softmax(target_logits + (static_cast<int64_t>(b) * (K + 1) + k) * V, pt);
      softmax(draft_logits + (static_cast<int64_t>(b) * K + k) * V, pd);
      const int x = drafts[b * K + k];
      if (static_cast<double>(u_accept[b * K + k]) * pd[x] < pt[x]) continue;
      for (int v = 0; v < V; ++v) r[v] = std::max(0.0, pt[v] - pd[v]);
      next_token[b] = draw(r, u_sample[b]);
      break;
    }
    n_accept[b] = k;
    if (k == K) {
      softmax(target_logits + (static_cast<int64_t>(b) * (K + 1) + K) * V, pt);
      next_token[b] = draw(pt, u_sample[b]);
    }
  }
}

}  // extern "C"
