// Two-stage beam candidate selection on sm_103a (article "SLM 生成式高并发推理引擎：
// 延迟约束下的有效吞吐优化", section 3.3):
//
//   BF16 logits [W_in, V] -> per beam the 2W largest logits (token ids; lowest
//   id on equal logits) -> scores read from the FP32 log-softmax over the full
//   vocabulary, plus the beam's cumulative score -> flatten W_in x 2W -> the
//   global 2W best (higher score first; equal scores by lower flat index,
//   i.e. lower parent, then the beam's own candidate order) with parents.
//
// One kernel, one read of the logits.  CTA (c, b) streams chunk c of beam b
// from HBM into registers (16-byte loads), computes the chunk's max and sum of
// exp in fp32, and keeps the chunk's exact top-2W.  Pruning at chunk level is
// safe for the same reason it is at beam level: a logit outside its chunk's
// top 2W has at least 2W better logits in its own beam.  The last CTA of a beam
// (an atomic ticket, no spinning) merges the chunks into the beam's FP32 log
// normaliser and its sorted top-2W with scores; the last beam to finish picks
// the global candidates from those sorted lists.
#include <algorithm>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "slm_internal.h"

namespace slm {
namespace sel {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxVec = 8;                       // 16-byte vectors per thread
constexpr int kMaxChunk = kThreads * kMaxVec * 8;  // 32768 logits per CTA
constexpr int kCap = 8192;                       // candidate slots in shared memory
constexpr float kLog2e = 1.4426950408889634f;

struct Shared {
  unsigned long long keys[kCap];
  int hist[256];
  int warp_i[kWarps];
  float warp_f[kWarps];
  unsigned long long kth;
  int k_rem;
  int count;
  int flag;
  float f0;
};

// ---------------------------------------------------------------------------
// Order-preserving keys
// ---------------------------------------------------------------------------
// bf16 bit pattern -> uint16 whose unsigned order is the value order; -0 maps
// to +0 so equal values compare equal.
__device__ __forceinline__ uint32_t bf16_key(uint32_t bits) {
  bits &= 0xFFFFu;
  if (bits == 0x8000u) bits = 0;
  return (bits & 0x8000u) ? (~bits & 0xFFFFu) : (bits | 0x8000u);
}

__device__ __forceinline__ uint32_t key_to_bf16(uint32_t key) {
  return (key & 0x8000u) ? (key & 0x7FFFu) : (~key & 0xFFFFu);
}

__device__ __forceinline__ uint32_t f32_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits) { return __uint_as_float((bits & 0xFFFFu) << 16); }

// Beam-local candidate key: larger = earlier (higher logit, then lower id).
__device__ __forceinline__ unsigned long long local_key(uint32_t bits, uint32_t token) {
  return (static_cast<unsigned long long>(bf16_key(bits)) << 32) | (0xFFFFFFFFu - token);
}

// Global candidate key: higher score, then lower parent, then lower rank in
// the parent's sorted list (= higher logit, then lower id).
__device__ __forceinline__ unsigned long long global_key(float score, uint32_t parent, uint32_t rank) {
  return (static_cast<unsigned long long>(f32_key(score)) << 32) | ((0xFFFFu - parent) << 16) | (0xFFFFu - rank);
}

// ---------------------------------------------------------------------------
// Block primitives
// ---------------------------------------------------------------------------
__device__ __forceinline__ float block_max(float v, Shared& sh) {
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int w = threadIdx.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sh.warp_f[w] = v;
  __syncthreads();
  float r = sh.warp_f[0];
  for (int i = 1; i < kWarps; ++i) r = fmaxf(r, sh.warp_f[i]);
  return r;
}

__device__ __forceinline__ float block_sum(float v, Shared& sh) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sh.warp_f[w] = v;
  __syncthreads();
  float r = 0.f;
  for (int i = 0; i < kWarps; ++i) r += sh.warp_f[i];  // fixed order: deterministic
  return r;
}

// Exclusive prefix sum of one int per thread; returns the total through *total.
__device__ __forceinline__ int block_exclusive_scan(int v, int* total, Shared& sh) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int x = v;
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();
  if (lane == 31) sh.warp_i[w] = x;
  __syncthreads();
  int base = 0, tot = 0;
  for (int i = 0; i < kWarps; ++i) {
    if (i < w) base += sh.warp_i[i];
    tot += sh.warp_i[i];
  }
  *total = tot;
  return base + x - v;
}

// Warp 0 finds, from the 256-bin histogram, the bin holding the k-th largest
// key (bins scanned from 255 down) and stores digit / remaining rank.
__device__ __forceinline__ void pick_bin(Shared& sh, int k, int* digit_out) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    // lane l owns bins [255 - 8l - 7, 255 - 8l], walked from the top
    int local[8];
    int s = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      local[i] = sh.hist[255 - 8 * lane - i];
      s += local[i];
    }
    int incl = s;
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const int excl = incl - s;
    const bool mine = (excl < k) && (incl >= k);
    const unsigned ball = __ballot_sync(0xffffffffu, mine);
    const int owner = ball ? (__ffs(ball) - 1) : 31;
    if (lane == owner) {
      int cum = excl, d = 255 - 8 * lane;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (cum + local[i] >= k) {
          d = 255 - 8 * lane - i;
          break;
        }
        cum += local[i];
      }
      *digit_out = d;
      sh.k_rem = k - cum;
    }
  }
}

// k-th largest (1-based) of the distinct 64-bit keys produced by key_at(i),
// i in [0, n), with the key's bits above `top_bit` all zero.  Radix select with
// 8-bit digits from the top; only keys matching the digits fixed so far take
// part in later passes.  Warp-aggregated histogram updates keep heavily tied
// inputs from serialising on one counter.
template <class KeyAt>
__device__ unsigned long long block_kth_largest(KeyAt key_at, int n, int k, int top_bit, Shared& sh) {
  unsigned long long prefix = 0, mask = 0;
  int shift = ((top_bit + 1 + 7) / 8) * 8 - 8;
  for (; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += kThreads) sh.hist[i] = 0;
    __syncthreads();
    const int n_round = (n + kThreads - 1) / kThreads * kThreads;
    for (int i = threadIdx.x; i < n_round; i += kThreads) {
      int digit = -1;
      if (i < n) {
        const unsigned long long key = key_at(i);
        if ((key & mask) == prefix) digit = static_cast<int>((key >> shift) & 255ull);
      }
      const unsigned peers = __match_any_sync(0xffffffffu, digit);
      if (digit >= 0 && (threadIdx.x & 31) == (__ffs(peers) - 1)) atomicAdd(&sh.hist[digit], __popc(peers));
    }
    __syncthreads();
    int* digit_slot = &sh.count;
    pick_bin(sh, k, digit_slot);
    __syncthreads();
    prefix |= static_cast<unsigned long long>(sh.count) << shift;
    mask |= 255ull << shift;
    k = sh.k_rem;
    __syncthreads();
  }
  return prefix;
}

// Descending bitonic sort of sh.keys[0, n_pow2) (n_pow2 a power of two).
__device__ void block_sort_desc(unsigned long long* keys, int n_pow2) {
  for (int size = 2; size <= n_pow2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      __syncthreads();
      for (int t = threadIdx.x; t < n_pow2 / 2; t += kThreads) {
        const int lo = 2 * t - (t & (stride - 1));
        const int hi = lo + stride;
        const bool desc = ((lo & size) == 0);
        const unsigned long long a = keys[lo], b = keys[hi];
        if ((a < b) == desc) {
          keys[lo] = b;
          keys[hi] = a;
        }
      }
    }
  }
  __syncthreads();
}

__device__ __forceinline__ int next_pow2(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
struct Params {
  const uint16_t* logits;  // [W_in, V] bf16 bits
  const float* cum;        // [W_in]
  int W_in, V, K;          // K = 2W candidates per beam and globally
  int W;
  int n_chunks, chunk;     // chunks per beam, logits per chunk (multiple of 8)
  bool vec_ok;             // 16-byte loads allowed
  // workspace
  unsigned long long* chunk_keys;  // [W_in, n_chunks, K]
  int* chunk_count;                // [W_in, n_chunks]
  float* chunk_m;                  // [W_in, n_chunks]
  float* chunk_l;                  // [W_in, n_chunks]
  float* row_score;                // [W_in, K] sorted
  int* row_token;                  // [W_in, K]
  int* row_count;                  // [W_in]
  unsigned* tickets;               // [W_in + 1], zero at launch
  float* row_lse;                  // [W_in]
  // outputs
  int32_t* out_token;
  int32_t* out_parent;
  float* out_score;
  int32_t* out_cand_token;
  int32_t* out_cand_parent;
  float* out_cand_score;
  float* out_lse;
};

__device__ void chunk_stage(const Params& p, Shared& sh, int b, int c);
__device__ void beam_stage(const Params& p, Shared& sh, int b);
__device__ void global_stage(const Params& p, Shared& sh);

__global__ void __launch_bounds__(kThreads, 2) beam_select_kernel(const Params p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  Shared& sh = *reinterpret_cast<Shared*>(smem_raw);
  const int c = blockIdx.x, b = blockIdx.y;

  chunk_stage(p, sh, b, c);

  // Ticket: the last chunk of beam b merges the beam.
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) sh.flag = (atomicAdd(&p.tickets[b], 1u) == static_cast<unsigned>(p.n_chunks - 1));
  __syncthreads();
  if (!sh.flag) return;
  __threadfence();
  beam_stage(p, sh, b);

  // Ticket: the last beam to be merged picks the global candidates.
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) sh.flag = (atomicAdd(&p.tickets[p.W_in], 1u) == static_cast<unsigned>(p.W_in - 1));
  __syncthreads();
  if (!sh.flag) return;
  __threadfence();
  global_stage(p, sh);
}

// Chunk c of beam b: partial (max, sum exp) and the chunk's exact top-K.
__device__ void chunk_stage(const Params& p, Shared& sh, int b, int c) {
  const int beg = c * p.chunk;
  const int n = min(p.V - beg, p.chunk);
  const uint16_t* src = p.logits + static_cast<int64_t>(b) * p.V + beg;

  // element e of vector i of this thread sits at index (i * kThreads + tid) * 8 + e
  uint4 reg[kMaxVec];
#pragma unroll
  for (int i = 0; i < kMaxVec; ++i) {
    const int idx = (i * kThreads + threadIdx.x) * 8;
    if (p.vec_ok && idx + 8 <= n) {
      reg[i] = __ldcs(reinterpret_cast<const uint4*>(src + idx));
    } else {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t lo = (idx + 2 * e < n) ? src[idx + 2 * e] : 0xFF80u;       // -inf padding
        const uint32_t hi = (idx + 2 * e + 1 < n) ? src[idx + 2 * e + 1] : 0xFF80u;
        w[e] = lo | (hi << 16);
      }
      reg[i] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }

  // chunk max
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < kMaxVec; ++i) {
    const uint32_t* w = reinterpret_cast<const uint32_t*>(&reg[i]);
#pragma unroll
    for (int e = 0; e < 4; ++e) mx = fmaxf(mx, fmaxf(bf16_bits_to_f32(w[e]), bf16_bits_to_f32(w[e] >> 16)));
  }
  const float m_c = block_max(mx, sh);

  const int K = min(p.K, n);
  // Candidate threshold from a sample (one logit per thread): a key low enough
  // that at least K logits of the chunk are at or above it with near
  // certainty, yet few enough to fit the candidate buffer.  If the guess
  // misses either way, the exact path over all logits runs instead.
  uint32_t tau = 0;  // take everything when the chunk is small
  if (n > kCap) {
    const int ns = min(kThreads, (n + 7) / 8);
    const int r_s = min(ns, (2 * K * ns + n - 1) / n + 16);
    sh.keys[threadIdx.x] = (threadIdx.x < ns) ? bf16_key(reinterpret_cast<const uint32_t*>(&reg[0])[0]) : 0ull;
    __syncthreads();
    const unsigned long long* sk = sh.keys;
    tau = static_cast<uint32_t>(block_kth_largest([&](int i) { return sk[i]; }, ns, r_s, 15, sh));
  }

  // sum of exp and candidate collection in one pass
  if (threadIdx.x == 0) sh.count = 0;
  __syncthreads();
  const float mref = m_c * kLog2e;
  float se = 0.f;
#pragma unroll
  for (int i = 0; i < kMaxVec; ++i) {
    const uint32_t* w = reinterpret_cast<const uint32_t*>(&reg[i]);
    const int idx = (i * kThreads + threadIdx.x) * 8;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const uint32_t bits = (e & 1) ? (w[e >> 1] >> 16) : (w[e >> 1] & 0xFFFFu);
      const float x = bf16_bits_to_f32(bits);
      se += exp2f(fmaf(x, kLog2e, -mref));
      const bool take = (idx + e < n) && (bf16_key(bits) >= tau);
      const unsigned ball = __ballot_sync(0xffffffffu, take);
      if (ball) {
        int base = 0;
        if ((threadIdx.x & 31) == __ffs(ball) - 1) base = atomicAdd(&sh.count, __popc(ball));
        base = __shfl_sync(0xffffffffu, base, __ffs(ball) - 1);
        if (take) {
          const int pos = base + __popc(ball & ((1u << (threadIdx.x & 31)) - 1u));
          if (pos < kCap) sh.keys[pos] = local_key(bits, static_cast<uint32_t>(beg + idx + e));
        }
      }
    }
  }
  const float l_c = block_sum(se, sh);  // contains __syncthreads
  const int m_cand = sh.count;

  unsigned long long* out = p.chunk_keys + (static_cast<int64_t>(b) * p.n_chunks + c) * p.K;
  if (m_cand >= K && m_cand <= kCap) {
    // exact top-K among the candidates
    const unsigned long long* sk = sh.keys;
    const unsigned long long kth = block_kth_largest([&](int i) { return sk[i]; }, m_cand, K, 47, sh);
    if (threadIdx.x == 0) sh.flag = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < m_cand; i += kThreads) {
      const unsigned long long key = sh.keys[i];
      if (key >= kth) out[atomicAdd(&sh.flag, 1)] = key;
    }
  } else {
    // exact top-K over every logit of the chunk, keys rebuilt from registers
    auto key_at = [&](int j) -> unsigned long long {
      // j enumerates (vector slot, element) of this thread: j = slot*8 + e
      const int i = j >> 3, e = j & 7;
      const int idx = (i * kThreads + threadIdx.x) * 8 + e;
      if (idx >= n) return 0ull;  // padding: below every real key
      const uint32_t* w = reinterpret_cast<const uint32_t*>(&reg[i]);
      const uint32_t bits = (e & 1) ? (w[e >> 1] >> 16) : (w[e >> 1] & 0xFFFFu);
      return local_key(bits, static_cast<uint32_t>(beg + idx));
    };
    // per-thread enumeration: each thread walks its own 64 slots; the generic
    // selector indexes i in [0, n) over threads, so adapt: slot = i / kThreads
    unsigned long long prefix = 0, mask = 0;
    int k = K;
    for (int shift = 40; shift >= 0; shift -= 8) {
      for (int i = threadIdx.x; i < 256; i += kThreads) sh.hist[i] = 0;
      __syncthreads();
#pragma unroll
      for (int j = 0; j < kMaxVec * 8; ++j) {
        const unsigned long long key = key_at(j);
        int digit = -1;
        if (key != 0ull && (key & mask) == prefix) digit = static_cast<int>((key >> shift) & 255ull);
        const unsigned peers = __match_any_sync(0xffffffffu, digit);
        if (digit >= 0 && (threadIdx.x & 31) == (__ffs(peers) - 1)) atomicAdd(&sh.hist[digit], __popc(peers));
      }
      __syncthreads();
      pick_bin(sh, k, &sh.count);
      __syncthreads();
      prefix |= static_cast<unsigned long long>(sh.count) << shift;
      mask |= 255ull << shift;
      k = sh.k_rem;
      __syncthreads();
    }
    if (threadIdx.x == 0) sh.flag = 0;
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kMaxVec * 8; ++j) {
      const unsigned long long key = key_at(j);
      if (key != 0ull && key >= prefix) out[atomicAdd(&sh.flag, 1)] = key;
    }
  }
  if (threadIdx.x == 0) {
    p.chunk_count[b * p.n_chunks + c] = K;
    p.chunk_m[b * p.n_chunks + c] = m_c;
    p.chunk_l[b * p.n_chunks + c] = l_c;
  }
}

// Beam b: FP32 log normaliser and the sorted top-K with scores.
__device__ void beam_stage(const Params& p, Shared& sh, int b) {
  // log-sum-exp from the chunk partials
  float m = -INFINITY;
  for (int c = 0; c < p.n_chunks; ++c) m = fmaxf(m, __ldcg(&p.chunk_m[b * p.n_chunks + c]));
  float l = 0.f;
  for (int c = 0; c < p.n_chunks; ++c)
    l += __ldcg(&p.chunk_l[b * p.n_chunks + c]) * exp2f((__ldcg(&p.chunk_m[b * p.n_chunks + c]) - m) * kLog2e);
  const float lse = m + logf(l);

  // gather every chunk's candidates
  int total = 0;
  for (int c = 0; c < p.n_chunks; ++c) {
    const int cnt = __ldcg(&p.chunk_count[b * p.n_chunks + c]);
    const unsigned long long* src = p.chunk_keys + (static_cast<int64_t>(b) * p.n_chunks + c) * p.K;
    for (int i = threadIdx.x; i < cnt; i += kThreads) sh.keys[total + i] = __ldcg(&src[i]);
    total += cnt;
  }
  __syncthreads();
  const int K = min(p.K, total);
  const unsigned long long* sk = sh.keys;
  const unsigned long long kth = block_kth_largest([&](int i) { return sk[i]; }, total, K, 47, sh);
  // compact the kept keys to the front (kept count is exactly K: keys are distinct)
  if (threadIdx.x == 0) sh.flag = 0;
  __syncthreads();
  unsigned long long mine[kCap / kThreads];
  int nm = 0;
  for (int i = threadIdx.x; i < total; i += kThreads) {
    const unsigned long long key = sh.keys[i];
    if (key >= kth) mine[nm++] = key;
  }
  __syncthreads();
  for (int i = 0; i < nm; ++i) sh.keys[atomicAdd(&sh.flag, 1)] = mine[i];
  const int n2 = next_pow2(K);
  __syncthreads();
  for (int i = K + threadIdx.x; i < n2; i += kThreads) sh.keys[i] = 0ull;
  block_sort_desc(sh.keys, n2);

  const float cum = p.cum[b];
  for (int r = threadIdx.x; r < K; r += kThreads) {
    const unsigned long long key = sh.keys[r];
    const uint32_t token = 0xFFFFFFFFu - static_cast<uint32_t>(key & 0xFFFFFFFFull);
    const float x = bf16_bits_to_f32(key_to_bf16(static_cast<uint32_t>(key >> 32)));
    const float lp = __fsub_rn(x, lse);      // FP32 log-probability
    p.row_score[static_cast<int64_t>(b) * p.K + r] = __fadd_rn(cum, lp);
    p.row_token[static_cast<int64_t>(b) * p.K + r] = static_cast<int>(token);
  }
  if (threadIdx.x == 0) {
    p.row_count[b] = K;
    p.row_lse[b] = lse;
    if (p.out_lse) p.out_lse[b] = lse;
  }
}

// Global top-K over the W_in sorted beam lists.
__device__ void global_stage(const Params& p, Shared& sh) {
  const int n_keep = p.K;
  const int W_in = p.W_in;
  // 1. sample the first c entries of every beam; the n_keep-th best sample is
  //    a lower bound of the n_keep-th best overall.
  const int per = min(p.K, max(1, 2 * ((n_keep + W_in - 1) / W_in)));
  const int n_s = W_in * per;  // <= kCap by construction (host checks)
  for (int i = threadIdx.x; i < n_s; i += kThreads) {
    const int b = i / per, r = i - b * per;
    const int cnt = __ldcg(&p.row_count[b]);
    sh.keys[i] = (r < cnt) ? global_key(__ldcg(&p.row_score[static_cast<int64_t>(b) * p.K + r]), b, r) : 0ull;
  }
  __syncthreads();
  const unsigned long long* sk = sh.keys;
  unsigned long long lo = block_kth_largest([&](int i) { return sk[i]; }, n_s, n_keep, 63, sh);

  // 2. count entries at or above the bound, per beam (lists are sorted, so a
  //    binary search per beam); raise the bound while they overflow.
  auto count_at_least = [&](unsigned long long bound) -> int {
    int local = 0;
    for (int b = threadIdx.x; b < W_in; b += kThreads) {
      int lo_i = 0, hi_i = __ldcg(&p.row_count[b]);  // first index with key < bound
      while (lo_i < hi_i) {
        const int mid = (lo_i + hi_i) >> 1;
        const unsigned long long k = global_key(__ldcg(&p.row_score[static_cast<int64_t>(b) * p.K + mid]), b, mid);
        if (k >= bound) lo_i = mid + 1;
        else hi_i = mid;
      }
      local += lo_i;
    }
    int tot;
    block_exclusive_scan(local, &tot, sh);
    return tot;
  };
  int m = count_at_least(lo);
  if (m > kCap) {
    // bisect the key range: count(bound) falls by at most 1 per key value,
    // so some bound has n_keep <= count <= kCap
    unsigned long long hi = ~0ull;
    while (true) {
      const unsigned long long mid = lo + (hi - lo) / 2;
      const int cm = count_at_least(mid);
      if (cm > kCap) lo = mid;
      else if (cm < n_keep) hi = mid;
      else { lo = mid; m = cm; break; }
    }
  }

  // 3. gather the entries >= lo
  int local = 0;
  for (int b = threadIdx.x; b < W_in; b += kThreads) {
    int lo_i = 0, hi_i = __ldcg(&p.row_count[b]);
    while (lo_i < hi_i) {
      const int mid = (lo_i + hi_i) >> 1;
      const unsigned long long k = global_key(__ldcg(&p.row_score[static_cast<int64_t>(b) * p.K + mid]), b, mid);
      if (k >= lo) lo_i = mid + 1;
      else hi_i = mid;
    }
    local += lo_i;
  }
  int tot;
  int off = block_exclusive_scan(local, &tot, sh);
  __syncthreads();
  for (int b = threadIdx.x; b < W_in; b += kThreads) {
    const int cnt = __ldcg(&p.row_count[b]);
    for (int r = 0; r < cnt; ++r) {
      const unsigned long long k = global_key(__ldcg(&p.row_score[static_cast<int64_t>(b) * p.K + r]), b, r);
      if (k < lo) break;
      sh.keys[off++] = k;
    }
  }
  __syncthreads();

  // 4. exact n_keep best, sorted
  const unsigned long long kth = block_kth_largest([&](int i) { return sk[i]; }, tot, n_keep, 63, sh);
  if (threadIdx.x == 0) sh.flag = 0;
  __syncthreads();
  unsigned long long mine[kCap / kThreads];
  int nm = 0;
  for (int i = threadIdx.x; i < tot; i += kThreads) {
    const unsigned long long key = sh.keys[i];
    if (key >= kth) mine[nm++] = key;
  }
  __syncthreads();
  for (int i = 0; i < nm; ++i) sh.keys[atomicAdd(&sh.flag, 1)] = mine[i];
  const int n2 = next_pow2(n_keep);
  __syncthreads();
  for (int i = n_keep + threadIdx.x; i < n2; i += kThreads) sh.keys[i] = 0ull;
  block_sort_desc(sh.keys, n2);

  for (int i = threadIdx.x; i < n_keep; i += kThreads) {
    const unsigned long long key = sh.keys[i];
    const int parent = 0xFFFF - static_cast<int>((key >> 16) & 0xFFFFull);
    const int rank = 0xFFFF - static_cast<int>(key & 0xFFFFull);
    const int token = __ldcg(&p.row_token[static_cast<int64_t>(parent) * p.K + rank]);
    const float score = __ldcg(&p.row_score[static_cast<int64_t>(parent) * p.K + rank]);
    if (i < p.W) {
      p.out_token[i] = token;
      p.out_parent[i] = parent;
      p.out_score[i] = score;
    }
    if (p.out_cand_token) p.out_cand_token[i] = token;
    if (p.out_cand_parent) p.out_cand_parent[i] = parent;
    if (p.out_cand_score) p.out_cand_score[i] = score;
  }
}

}  // namespace sel

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
namespace {

struct SelLayout {
  int n_chunks, chunk;
  size_t off_keys, off_count, off_m, off_l, off_rscore, off_rtoken, off_rcount, off_tickets, off_lse, total;
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

bool sel_layout(int W_in, int V, int W, SelLayout* L) {
  if (W_in <= 0 || V <= 0 || W <= 0) return false;
  const int K = 2 * W;
  // Chunks: at most kMaxChunk logits, enough CTAs to cover the GPU a few
  // times over, and few enough that one beam's candidates fit the buffer.
  int n_chunks = (V + sel::kMaxChunk - 1) / sel::kMaxChunk;
  const int target_ctas = 1216;  // 8 per SM on 152 SMs
  while (static_cast<int64_t>(n_chunks) * W_in < target_ctas && n_chunks * 2 * 8 <= V &&
         (n_chunks * 2) * static_cast<int64_t>(K) <= sel::kCap)
    n_chunks *= 2;
  int chunk = (V + n_chunks - 1) / n_chunks;
  chunk = (chunk + 7) / 8 * 8;
  n_chunks = (V + chunk - 1) / chunk;
  if (static_cast<int64_t>(n_chunks) * K > sel::kCap) return false;
  L->n_chunks = n_chunks;
  L->chunk = chunk;
  size_t o = 0;
  L->off_keys = o;    o = align256(o + sizeof(unsigned long long) * size_t(W_in) * n_chunks * K);
  L->off_count = o;   o = align256(o + sizeof(int) * size_t(W_in) * n_chunks);
  L->off_m = o;       o = align256(o + sizeof(float) * size_t(W_in) * n_chunks);
  L->off_l = o;       o = align256(o + sizeof(float) * size_t(W_in) * n_chunks);
  L->off_rscore = o;  o = align256(o + sizeof(float) * size_t(W_in) * K);
  L->off_rtoken = o;  o = align256(o + sizeof(int) * size_t(W_in) * K);
  L->off_rcount = o;  o = align256(o + sizeof(int) * size_t(W_in));
  L->off_tickets = o; o = align256(o + sizeof(unsigned) * size_t(W_in + 1));
  L->off_lse = o;     o = align256(o + sizeof(float) * size_t(W_in));
  L->total = o;
  return true;
}

}  // namespace

size_t beam_select_workspace_bytes(int W_in, int V, int W) {
  SelLayout L;
  if (!sel_layout(W_in, V, W, &L)) return 0;
  return L.total;
}

bool beam_select_supported(int W_in, int V, int W) {
  SelLayout L;
  if (!sel_layout(W_in, V, W, &L)) return false;
  // the global stage samples 2 * ceil(2W / W_in) entries of every beam
  const int K = 2 * W;
  const int per = std::min(K, std::max(1, 2 * ((K + W_in - 1) / W_in)));
  return static_cast<int64_t>(W_in) * per <= sel::kCap && K <= sel::kCap / 2 && W_in <= 0xFFFF && K <= 0xFFFF;
}

cudaError_t launch_beam_select(const void* logits, const float* cum, int W_in, int V, int W, int32_t* out_token,
                               int32_t* out_parent, float* out_score, int32_t* out_cand_token,
                               int32_t* out_cand_parent, float* out_cand_score, float* out_lse, void* workspace,
                               cudaStream_t stream) {
  SelLayout L;
  if (!sel_layout(W_in, V, W, &L)) return cudaErrorInvalidValue;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  sel::Params p{};
  p.logits = static_cast<const uint16_t*>(logits);
  p.cum = cum;
  p.W_in = W_in;
  p.V = V;
  p.K = 2 * W;
  p.W = W;
  p.n_chunks = L.n_chunks;
  p.chunk = L.chunk;
  p.vec_ok = (V % 8 == 0) && ((reinterpret_cast<uintptr_t>(logits) & 15) == 0);
  p.chunk_keys = reinterpret_cast<unsigned long long*>(ws + L.off_keys);
  p.chunk_count = reinterpret_cast<int*>(ws + L.off_count);
  p.chunk_m = reinterpret_cast<float*>(ws + L.off_m);
  p.chunk_l = reinterpret_cast<float*>(ws + L.off_l);
  p.row_score = reinterpret_cast<float*>(ws + L.off_rscore);
  p.row_token = reinterpret_cast<int*>(ws + L.off_rtoken);
  p.row_count = reinterpret_cast<int*>(ws + L.off_rcount);
  p.tickets = reinterpret_cast<unsigned*>(ws + L.off_tickets);
  p.row_lse = reinterpret_cast<float*>(ws + L.off_lse);
  p.out_token = out_token;
  p.out_parent = out_parent;
  p.out_score = out_score;
  p.out_cand_token = out_cand_token;
  p.out_cand_parent = out_cand_parent;
  p.out_cand_score = out_cand_score;
  p.out_lse = out_lse;

  cudaError_t e = cudaMemsetAsync(p.tickets, 0, sizeof(unsigned) * size_t(W_in + 1), stream);
  if (e != cudaSuccess) return e;
  const size_t smem = sizeof(sel::Shared);
  e = cudaFuncSetAttribute(sel::beam_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(L.n_chunks, W_in);
  sel::beam_select_kernel<<<grid, sel::kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace slm
