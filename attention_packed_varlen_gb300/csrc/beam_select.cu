// Two-stage beam candidate selection on sm_103a (article "SLM 生成式高并发推理引擎：
// 延迟约束下的有效吞吐优化", section 3.3):
//
//   BF16 logits [W_in, V] -> per beam the 2W largest logits (token ids; lowest
//   id on equal logits) -> scores read from the FP32 log-softmax over the full
//   vocabulary, plus the beam's cumulative score -> flatten W_in x 2W -> the
//   global 2W best (higher score first; equal scores by lower flat index,
//   i.e. lower parent, then the beam's own candidate order) with parents.
//
// Three kernels, one read of the logits.
//
// 1. threshold (one CTA per beam): histograms 4096 sampled logits (64-byte
//    runs spread over the row) by the top 12 bits of an order-preserving key
//    and picks a candidate threshold tau_b that keeps the beam's 2W best with
//    near certainty while passing only a few percent of the row.
// 2. stream (CTA (c, b) = chunk c of beam b): the HBM pass.  16-byte loads
//    into registers, chunk max on packed bf16, fp32 sum of exp2 (MUFU)
//    against it, and a count of logits >= tau_b; one atomic per CTA reserves
//    room in the beam's candidate buffer and the candidates are written
//    there.  Small and spill-free so several CTAs share an SM.
// 3. merge (one CTA per beam): FP32 log normaliser from the chunk partials,
//    the exact top-2W of the beam's candidates (a missed threshold falls back
//    to an exact scan of the row), sorted, with scores.  The last beam to
//    finish (atomic ticket, no spinning) picks the global candidates from the
//    sorted beam lists.
//
// Selections are radix selects whose 8-bit digits are taken relative to the
// live key range, so clustered keys still spread over the bins of the
// per-warp shared-memory histograms, and a select stops as soon as the bin it
// follows holds a single key.
#include <algorithm>
#include <cfloat>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "slm_internal.h"

namespace slm {
namespace sel {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxVec = 4;                        // 16-byte vectors per thread
constexpr int kMaxChunk = kThreads * kMaxVec * 8; // 16384 logits per stream CTA
constexpr int kCap = 8192;                        // candidate keys per beam
constexpr int kThrThreads = 256;                  // threshold kernel
constexpr int kThrBins = 4096;                    // top 12 bits of the 16-bit key
constexpr int kSampleRuns = 128;                  // runs of 32 logits sampled per beam
constexpr int kSelCap = 2048;                     // selected keys: 2W <= 2048
constexpr float kLog2e = 1.4426950408889634f;

struct Shared {
  unsigned long long keys[kCap];
  unsigned long long sel[kSelCap];
  int whist[kWarps][256];
  int hist[256];
  unsigned long long warp_u64[2][kWarps];
  int warp_i[kWarps];
  float warp_f[kWarps];
  unsigned long long u64;
  int digit, k_rem, above, in_bin, counter, flag, base;
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

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits) { return __uint_as_float((bits & 0xFFFFu) << 16); }

__device__ __forceinline__ uint32_t f32_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Beam-local candidate key: larger = earlier (higher logit, then lower id).
__device__ __forceinline__ unsigned long long local_key(uint32_t key16, uint32_t token) {
  return (static_cast<unsigned long long>(key16) << 32) | (0xFFFFFFFFu - token);
}

// Global candidate key: higher score, then lower parent, then lower rank in
// the parent's sorted list (= higher logit, then lower id).
__device__ __forceinline__ unsigned long long global_key(float score, uint32_t parent, uint32_t rank) {
  return (static_cast<unsigned long long>(f32_key(score)) << 32) | ((0xFFFFu - parent) << 16) | (0xFFFFu - rank);
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Shared memory of the stream kernel: reductions only.
struct Small {
  int warp_i[kWarps];
  float warp_f[kWarps];
  int base;
};

// ---------------------------------------------------------------------------
// Block primitives (every thread of the CTA calls them)
// ---------------------------------------------------------------------------
template <class S>
__device__ __forceinline__ float block_max(float v, S& sh) {
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sh.warp_f[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = sh.warp_f[0];
  for (int i = 1; i < kWarps; ++i) r = fmaxf(r, sh.warp_f[i]);
  return r;
}

template <class S>
__device__ __forceinline__ float block_sum(float v, S& sh) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sh.warp_f[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = 0.f;
  for (int i = 0; i < kWarps; ++i) r += sh.warp_f[i];  // fixed order: deterministic
  return r;
}

// Exclusive prefix sum of one int per thread (thread order); *total = sum.
template <class S>
__device__ __forceinline__ int block_exclusive_scan(int v, int* total, S& sh) {
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

__device__ __forceinline__ void block_minmax(unsigned long long& mn, unsigned long long& mx, Shared& sh) {
  for (int o = 16; o > 0; o >>= 1) {
    mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  __syncthreads();
  if ((threadIdx.x & 31) == 0) {
    sh.warp_u64[0][threadIdx.x >> 5] = mn;
    sh.warp_u64[1][threadIdx.x >> 5] = mx;
  }
  __syncthreads();
  mn = ~0ull;
  mx = 0ull;
  for (int i = 0; i < kWarps; ++i) {
    mn = min(mn, sh.warp_u64[0][i]);
    mx = max(mx, sh.warp_u64[1][i]);
  }
}

__device__ __forceinline__ void hist_clear(Shared& sh) {
  int* h = &sh.whist[0][0];
  for (int i = threadIdx.x; i < kWarps * 256; i += kThreads) h[i] = 0;
}

__device__ __forceinline__ void hist_add(Shared& sh, uint32_t digit) {
  atomicAdd(&sh.whist[threadIdx.x >> 5][digit], 1);
}

// Sums the per-warp histograms, then warp 0 finds the bin holding the k-th
// largest item (bins walked from 255 down): digit, items above the bin, items
// in it, and the rank left inside it.  Ends with all results visible.
__device__ __forceinline__ void hist_pick(Shared& sh, int k) {
  __syncthreads();
  if (threadIdx.x < 256) {
    int s = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) s += sh.whist[w][threadIdx.x];
    sh.hist[threadIdx.x] = s;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
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
    const unsigned ball = __ballot_sync(0xffffffffu, excl < k && incl >= k);
    const int owner = ball ? (__ffs(ball) - 1) : 31;
    if (lane == owner) {
      int cum = excl, d = 255 - 8 * lane, in_bin = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (cum + local[i] >= k) {
          d = 255 - 8 * lane - i;
          in_bin = local[i];
          break;
        }
        cum += local[i];
      }
      sh.digit = d;
      sh.above = cum;
      sh.in_bin = in_bin;
      sh.k_rem = k - cum;
    }
  }
  __syncthreads();
}

// k-th largest (1-based) of the distinct 64-bit keys every thread visits with
// for_each(f) (f(key)).  Each pass histograms the keys still in the live range
// [lo, hi] by the 8 bits just below the range's leading bit, then narrows the
// range to the bin holding the k-th key; a bin with a single key ends it.
template <class ForEach>
__device__ unsigned long long block_kth(ForEach for_each, int k, Shared& sh) {
  unsigned long long lo = ~0ull, hi = 0ull;
  for_each([&](unsigned long long key) {
    lo = min(lo, key);
    hi = max(hi, key);
  });
  block_minmax(lo, hi, sh);
  while (lo < hi) {
    const unsigned long long span = hi - lo;
    const int s = max(0, 64 - __clzll(span) - 8);
    hist_clear(sh);
    __syncthreads();
    const unsigned long long lo_c = lo, hi_c = hi;
    for_each([&](unsigned long long key) {
      if (key >= lo_c && key <= hi_c) hist_add(sh, static_cast<uint32_t>((key - lo_c) >> s));
    });
    hist_pick(sh, k);
    const unsigned long long base = lo + (static_cast<unsigned long long>(sh.digit) << s);
    const unsigned long long width = (1ull << s) - 1;
    hi = (hi - base <= width) ? hi : base + width;
    lo = base;
    k = sh.k_rem;
    const int in_bin = sh.in_bin;
    __syncthreads();
    if (in_bin == 1 && lo < hi) {
      const unsigned long long lo_b = lo, hi_b = hi;
      for_each([&](unsigned long long key) {
        if (key >= lo_b && key <= hi_b) sh.u64 = key;
      });
      __syncthreads();
      const unsigned long long r = sh.u64;
      __syncthreads();
      return r;
    }
  }
  return lo;
}

// Descending bitonic sort of keys[0, n_pow2).
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
// The kernels
// ---------------------------------------------------------------------------
struct Params {
  const uint16_t* logits;  // [W_in, V] bf16 bits
  const float* cum;        // [W_in]
  int W_in, V, K;          // K = 2W candidates per beam and globally
  int W;
  int n_chunks, chunk;     // chunks per beam, logits per chunk (multiple of 8)
  int sample_per;          // entries of each beam the global stage samples
  bool vec_ok;             // 16-byte loads allowed
  // workspace
  float* tau;                      // [W_in] candidate threshold per beam
  int* cand_count;                 // [W_in]
  unsigned long long* cand_keys;   // [W_in, kCap]
  float* chunk_m;                  // [W_in, n_chunks]
  float* chunk_l;                  // [W_in, n_chunks]
  float* row_score;                // [W_in, K] sorted
  int* row_token;                  // [W_in, K]
  unsigned* tickets;               // [W_in + 1]
  // outputs
  int32_t* out_token;
  int32_t* out_parent;
  float* out_score;
  int32_t* out_cand_token;
  int32_t* out_cand_parent;
  float* out_cand_score;
  float* out_lse;
};

// Beam b's candidate threshold from a sample of its logits; also resets the
// beam's counter and tickets for the stream kernel that follows.
__global__ void __launch_bounds__(kThrThreads) threshold_kernel(const Params p) {
  __shared__ int hist[kThrBins];
  __shared__ int warp_tot[kThrThreads / 32];
  const int b = blockIdx.x;
  if (threadIdx.x == 0) {
    p.cand_count[b] = 0;
    p.tickets[b] = 0;
    if (b == 0) p.tickets[p.W_in] = 0;
  }
  const uint16_t* row = p.logits + static_cast<int64_t>(b) * p.V;
  // A beam small enough to fit the candidate buffer keeps everything.
  if (p.V <= kCap) {
    if (threadIdx.x == 0) p.tau[b] = -INFINITY;
    return;
  }
  for (int i = threadIdx.x; i < kThrBins; i += kThrThreads) hist[i] = 0;
  __syncthreads();
  // runs of 32 consecutive logits at evenly spaced starts
  const int ns = kSampleRuns * 32;
  const int64_t stride = (static_cast<int64_t>(p.V) - 32) / (kSampleRuns - 1);
  for (int s = threadIdx.x; s < ns; s += kThrThreads) {
    const int64_t idx = (s >> 5) * stride + (s & 31);
    atomicAdd(&hist[bf16_key(row[idx]) >> 4], 1);
  }
  __syncthreads();
  const float expect = static_cast<float>(p.K) * ns / p.V;
  const int r = min(ns, static_cast<int>(ceilf(expect + 6.f * sqrtf(expect) + 8.f)));
  // the bin holding the r-th largest sample (bins walked from the top)
  constexpr int kPer = kThrBins / kThrThreads;  // 16 bins per thread, highest first
  const int first = kThrBins - 1 - kPer * threadIdx.x;
  int sum = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) sum += hist[first - i];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int x = sum;
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[w] = x;
  __syncthreads();
  int before = x - sum;
  for (int i = 0; i < w; ++i) before += warp_tot[i];
  if (before < r && before + sum >= r) {
    int cum = before, bin = first;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      cum += hist[first - i];
      if (cum >= r) {
        bin = first - i;
        break;
      }
    }
    // lower edge of the bin: every logit of the bin passes
    p.tau[b] = bf16_bits_to_f32(key_to_bf16(static_cast<uint32_t>(bin) << 4));
  }
}

__device__ void beam_merge(const Params& p, Shared& sh, int b);
__device__ void global_stage(const Params& p, Shared& sh);

__global__ void __launch_bounds__(kThreads, 2) stream_kernel(const Params p) {
  __shared__ Small sh;
  const int c = blockIdx.x, b = blockIdx.y;
  const int beg = c * p.chunk;
  const int n = min(p.V - beg, p.chunk);
  const uint16_t* src = p.logits + static_cast<int64_t>(b) * p.V + beg;

  // element e of vector i of this thread sits at chunk index (i * kThreads + tid) * 8 + e
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
        const uint32_t lo = (idx + 2 * e < n) ? src[idx + 2 * e] : 0xFF80u;  // -inf padding
        const uint32_t hi = (idx + 2 * e + 1 < n) ? src[idx + 2 * e + 1] : 0xFF80u;
        w[e] = lo | (hi << 16);
      }
      reg[i] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
  auto word = [&](int i, int h) -> uint32_t {
    return h == 0 ? reg[i].x : h == 1 ? reg[i].y : h == 2 ? reg[i].z : reg[i].w;
  };

  // chunk max on packed bf16 pairs (exact)
  __nv_bfloat162 m2 = __float2bfloat162_rn(-INFINITY);
#pragma unroll
  for (int i = 0; i < kMaxVec; ++i)
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const uint32_t w = word(i, h);
      m2 = __hmax2(m2, *reinterpret_cast<const __nv_bfloat162*>(&w));
    }
  const float m_c = block_max(fmaxf(__low2float(m2), __high2float(m2)), sh);

  // one pass: sum of exp against the chunk max, and the candidate count
  const float tau = p.tau[b];
  const float mref = m_c * kLog2e;
  float se = 0.f;
  int cnt = 0;
#pragma unroll
  for (int i = 0; i < kMaxVec; ++i) {
    const int idx = (i * kThreads + threadIdx.x) * 8;
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const uint32_t w = word(i, h);
      const float x0 = __uint_as_float(w << 16), x1 = __uint_as_float(w & 0xFFFF0000u);
      se += ex2(fmaf(x0, kLog2e, -mref)) + ex2(fmaf(x1, kLog2e, -mref));
      cnt += (x0 >= tau && idx + 2 * h < n) + (x1 >= tau && idx + 2 * h + 1 < n);
    }
  }
  const float l_c = block_sum(se, sh);
  int total;
  int off = block_exclusive_scan(cnt, &total, sh);
  if (threadIdx.x == 0) sh.base = atomicAdd(&p.cand_count[b], total);
  __syncthreads();
  off += sh.base;
  unsigned long long* cand = p.cand_keys + static_cast<int64_t>(b) * kCap;
  if (cnt > 0) {
#pragma unroll
    for (int i = 0; i < kMaxVec; ++i) {
      const int idx = (i * kThreads + threadIdx.x) * 8;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const uint32_t w = word(i, e >> 1);
        const uint32_t bits = (e & 1) ? (w >> 16) : (w & 0xFFFFu);
        if (bf16_bits_to_f32(bits) >= tau && idx + e < n) {
          if (off < kCap) cand[off] = local_key(bf16_key(bits), static_cast<uint32_t>(beg + idx + e));
          ++off;
        }
      }
    }
  }
  if (threadIdx.x == 0) {
    p.chunk_m[b * p.n_chunks + c] = m_c;
    p.chunk_l[b * p.n_chunks + c] = l_c;
  }
}

__global__ void __launch_bounds__(kThreads, 1) merge_kernel(const Params p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  Shared& sh = *reinterpret_cast<Shared*>(smem_raw);
  const int b = blockIdx.x;
  beam_merge(p, sh, b);

  // Ticket: the last beam to be merged picks the global candidates.
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) sh.flag = (atomicAdd(&p.tickets[p.W_in], 1u) == static_cast<unsigned>(p.W_in - 1));
  __syncthreads();
  if (!sh.flag) return;
  __threadfence();
  global_stage(p, sh);
}

// Beam b: FP32 log normaliser and the sorted top-K with scores
// fl32(cum + fl32(x - lse)).
__device__ void beam_merge(const Params& p, Shared& sh, int b) {
  const int K = p.K;
  float m = -INFINITY;
  for (int c = 0; c < p.n_chunks; ++c) m = fmaxf(m, __ldcg(&p.chunk_m[b * p.n_chunks + c]));
  float l = 0.f;
  for (int c = 0; c < p.n_chunks; ++c)
    l += __ldcg(&p.chunk_l[b * p.n_chunks + c]) * ex2((__ldcg(&p.chunk_m[b * p.n_chunks + c]) - m) * kLog2e);
  const float lse = m + logf(l);

  const int c_b = __ldcg(&p.cand_count[b]);
  if (c_b >= K && c_b <= kCap) {
    const unsigned long long* cand = p.cand_keys + static_cast<int64_t>(b) * kCap;
    for (int i = threadIdx.x; i < c_b; i += kThreads) sh.keys[i] = __ldcg(&cand[i]);
    __syncthreads();
    auto for_each_cand = [&](auto f) {
      for (int i = threadIdx.x; i < c_b; i += kThreads) f(sh.keys[i]);
    };
    const unsigned long long kth = block_kth(for_each_cand, K, sh);
    if (threadIdx.x == 0) sh.counter = 0;
    __syncthreads();
    for_each_cand([&](unsigned long long key) {
      if (key >= kth) sh.sel[atomicAdd(&sh.counter, 1)] = key;
    });
  } else {
    // The threshold missed (rare: a freak sample, heavy ties or -inf
    // logits): exact top-K over the whole row.
    const uint16_t* row = p.logits + static_cast<int64_t>(b) * p.V;
    auto for_each_row = [&](auto f) {
      for (int j = threadIdx.x; j < p.V; j += kThreads) f(local_key(bf16_key(row[j]), static_cast<uint32_t>(j)));
    };
    const unsigned long long kth = block_kth(for_each_row, K, sh);
    if (threadIdx.x == 0) sh.counter = 0;
    __syncthreads();
    for_each_row([&](unsigned long long key) {
      if (key >= kth) sh.sel[atomicAdd(&sh.counter, 1)] = key;
    });
  }
  const int n2 = next_pow2(K);
  __syncthreads();
  for (int i = K + threadIdx.x; i < n2; i += kThreads) sh.sel[i] = 0ull;
  block_sort_desc(sh.sel, n2);

  const float cum = p.cum[b];
  for (int r = threadIdx.x; r < K; r += kThreads) {
    const unsigned long long key = sh.sel[r];
    const uint32_t token = 0xFFFFFFFFu - static_cast<uint32_t>(key & 0xFFFFFFFFull);
    const float x = bf16_bits_to_f32(key_to_bf16(static_cast<uint32_t>(key >> 32)));
    const float lp = __fsub_rn(x, lse);  // FP32 log-probability
    p.row_score[static_cast<int64_t>(b) * K + r] = __fadd_rn(cum, lp);
    p.row_token[static_cast<int64_t>(b) * K + r] = static_cast<int>(token);
  }
  if (threadIdx.x == 0 && p.out_lse) p.out_lse[b] = lse;
}

// Global top-K over the W_in sorted beam lists (each exactly K long).
__device__ void global_stage(const Params& p, Shared& sh) {
  const int n_keep = p.K;
  const int W_in = p.W_in;
  const int K = p.K;
  const int per = p.sample_per;  // W_in * per >= n_keep and <= kSelCap
  auto gkey = [&](int b, int r) {
    return global_key(__ldcg(&p.row_score[static_cast<int64_t>(b) * K + r]), b, r);
  };
  // 1. the first `per` entries of every beam; the n_keep-th best of them is a
  //    lower bound of the n_keep-th best overall
  const int n_s = W_in * per;
  for (int i = threadIdx.x; i < n_s; i += kThreads) sh.sel[i] = gkey(i / per, i % per);
  __syncthreads();
  auto for_each_sample = [&](auto f) {
    for (int i = threadIdx.x; i < n_s; i += kThreads) f(sh.sel[i]);
  };
  unsigned long long lo = block_kth(for_each_sample, n_keep, sh);

  // 2. entries at or above the bound, per beam: from the sample, and past it
  //    by binary search in the beam's sorted list when the whole sample clears
  auto count_global = [&](int b, unsigned long long bound, int from) {
    int lo_i = from, hi_i = K;
    while (lo_i < hi_i) {
      const int mid = (lo_i + hi_i) >> 1;
      if (gkey(b, mid) >= bound) lo_i = mid + 1;
      else hi_i = mid;
    }
    return lo_i;
  };
  auto beam_count = [&](int b, unsigned long long bound) {
    int c = 0;
    while (c < per && sh.sel[b * per + c] >= bound) ++c;
    if (c == per && per < K) c = count_global(b, bound, per);
    return c;
  };
  constexpr int kBeamsPerThread = 2;  // W_in <= 1024
  int cnt[kBeamsPerThread];
  int mine = 0;
#pragma unroll
  for (int j = 0; j < kBeamsPerThread; ++j) {
    const int b = threadIdx.x + j * kThreads;
    cnt[j] = (b < W_in) ? beam_count(b, lo) : 0;
    mine += cnt[j];
  }
  int m;
  int off = block_exclusive_scan(mine, &m, sh);
  if (m > kCap) {
    // Rare: bisect the key range; the count drops by at most one per key
    // value, so some bound keeps between n_keep and kCap entries.
    unsigned long long hi = ~0ull;
    while (true) {
      const unsigned long long mid = lo + (hi - lo) / 2;
      int part = 0;
      for (int b = threadIdx.x; b < W_in; b += kThreads) part += count_global(b, mid, 0);
      int cm;
      block_exclusive_scan(part, &cm, sh);
      if (cm > kCap) lo = mid;
      else if (cm < n_keep) hi = mid;
      else {
        lo = mid;
        break;
      }
    }
    mine = 0;
#pragma unroll
    for (int j = 0; j < kBeamsPerThread; ++j) {
      const int b = threadIdx.x + j * kThreads;
      cnt[j] = (b < W_in) ? count_global(b, lo, 0) : 0;
      mine += cnt[j];
    }
    off = block_exclusive_scan(mine, &m, sh);
  }

  // 3. gather the entries at or above the bound
#pragma unroll
  for (int j = 0; j < kBeamsPerThread; ++j) {
    const int b = threadIdx.x + j * kThreads;
    for (int r = 0; r < cnt[j]; ++r) sh.keys[off++] = (r < per) ? sh.sel[b * per + r] : gkey(b, r);
  }
  __syncthreads();

  // 4. exact n_keep best, sorted
  auto for_each_m = [&](auto f) {
    for (int i = threadIdx.x; i < m; i += kThreads) f(sh.keys[i]);
  };
  const unsigned long long kth = block_kth(for_each_m, n_keep, sh);
  if (threadIdx.x == 0) sh.counter = 0;
  __syncthreads();
  for_each_m([&](unsigned long long key) {
    if (key >= kth) sh.sel[atomicAdd(&sh.counter, 1)] = key;
  });
  const int n2 = next_pow2(n_keep);
  __syncthreads();
  for (int i = n_keep + threadIdx.x; i < n2; i += kThreads) sh.sel[i] = 0ull;
  block_sort_desc(sh.sel, n2);

  for (int i = threadIdx.x; i < n_keep; i += kThreads) {
    const unsigned long long key = sh.sel[i];
    const int parent = 0xFFFF - static_cast<int>((key >> 16) & 0xFFFFull);
    const int rank = 0xFFFF - static_cast<int>(key & 0xFFFFull);
    const int token = __ldcg(&p.row_token[static_cast<int64_t>(parent) * K + rank]);
    const float score = __ldcg(&p.row_score[static_cast<int64_t>(parent) * K + rank]);
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
  int n_chunks, chunk, sample_per;
  size_t off_tau, off_count, off_cand, off_m, off_l, off_rscore, off_rtoken, off_tickets, total;
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

bool sel_layout(int W_in, int V, int W, SelLayout* L) {
  if (W_in <= 0 || V <= 0 || W <= 0) return false;
  const int64_t K = 2 * static_cast<int64_t>(W);
  if (K > sel::kSelCap || K > V || W_in > 1024 || V >= (1 << 24)) return false;
  // Chunks: at most kMaxChunk logits, about 8 CTAs per SM over the grid
  // (152 SMs), and at least 4096 logits each.
  int n_chunks = std::max((V + sel::kMaxChunk - 1) / sel::kMaxChunk, (1216 + W_in / 2) / W_in);
  n_chunks = std::min(n_chunks, std::max((V + sel::kMaxChunk - 1) / sel::kMaxChunk, V / 4096));
  n_chunks = std::max(n_chunks, 1);
  int chunk = (V + n_chunks - 1) / n_chunks;
  chunk = (chunk + 7) / 8 * 8;
  n_chunks = (V + chunk - 1) / chunk;
  L->n_chunks = n_chunks;
  L->chunk = chunk;
  // global stage sample: as many entries per beam as fit, at least enough to
  // hold n_keep = K entries in total
  const int per = static_cast<int>(std::min<int64_t>(K, sel::kSelCap / W_in));
  if (static_cast<int64_t>(per) * W_in < K) return false;
  L->sample_per = per;
  size_t o = 0;
  L->off_tau = o;     o = align256(o + sizeof(float) * size_t(W_in));
  L->off_count = o;   o = align256(o + sizeof(int) * size_t(W_in));
  L->off_cand = o;    o = align256(o + sizeof(unsigned long long) * size_t(W_in) * sel::kCap);
  L->off_m = o;       o = align256(o + sizeof(float) * size_t(W_in) * n_chunks);
  L->off_l = o;       o = align256(o + sizeof(float) * size_t(W_in) * n_chunks);
  L->off_rscore = o;  o = align256(o + sizeof(float) * size_t(W_in) * K);
  L->off_rtoken = o;  o = align256(o + sizeof(int) * size_t(W_in) * K);
  L->off_tickets = o; o = align256(o + sizeof(unsigned) * size_t(W_in + 1));
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
  return sel_layout(W_in, V, W, &L);
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
  p.sample_per = L.sample_per;
  p.vec_ok = (V % 8 == 0) && ((reinterpret_cast<uintptr_t>(logits) & 15) == 0);
  p.tau = reinterpret_cast<float*>(ws + L.off_tau);
  p.cand_count = reinterpret_cast<int*>(ws + L.off_count);
  p.cand_keys = reinterpret_cast<unsigned long long*>(ws + L.off_cand);
  p.chunk_m = reinterpret_cast<float*>(ws + L.off_m);
  p.chunk_l = reinterpret_cast<float*>(ws + L.off_l);
  p.row_score = reinterpret_cast<float*>(ws + L.off_rscore);
  p.row_token = reinterpret_cast<int*>(ws + L.off_rtoken);
  p.tickets = reinterpret_cast<unsigned*>(ws + L.off_tickets);
  p.out_token = out_token;
  p.out_parent = out_parent;
  p.out_score = out_score;
  p.out_cand_token = out_cand_token;
  p.out_cand_parent = out_cand_parent;
  p.out_cand_score = out_cand_score;
  p.out_lse = out_lse;

  sel::threshold_kernel<<<W_in, sel::kThrThreads, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t smem = sizeof(sel::Shared);
  e = cudaFuncSetAttribute(sel::merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(L.n_chunks, W_in);
  sel::stream_kernel<<<grid, sel::kThreads, 0, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  sel::merge_kernel<<<W_in, sel::kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace slm
