// Two-stage beam candidate selection on sm_103a (article "SLM 生成式高并发推理引擎：
// 延迟约束下的有效吞吐优化", section 3.3):
//
//   BF16 logits [W_in, V] -> per beam the 2W largest logits (token ids; lowest
//   id on equal logits) -> scores read from the FP32 log-softmax over the full
//   vocabulary, plus the beam's cumulative score -> flatten W_in x 2W -> the
//   global 2W best (higher score first; equal scores by lower parent, then
//   higher logit, then lower id) with parents.
//
// The article's pruning claim (a token below rank 2W in its own beam cannot
// reach the global top 2W) is used the other way round: every beam hands the
// global stage a superset of its top 2W -- all of its logits at or above a
// threshold tau_b -- and the global stage ranks that superset with the full
// order.  The result is the same, and no per-beam sort is needed.
//
// Four kernels, one read of the logits from HBM; each later kernel is
// launched as a programmatic dependent of the one before, so it is resident
// and waiting (griddepcontrol.wait) when its predecessor ends:
//
// 1. prep (one CTA per beam): resets the per-call counters and the score
//    histogram, and from 4096 sampled logits picks tau_b (keeps the beam's 2W
//    best with near certainty while passing ~1.5% of the row) and a softmax
//    reference R_b (the sample maximum).
// 2. stream (persistent, one CTA per SM): a producer warp streams 16 KB tiles
//    of the logits into an 8-stage shared-memory ring with 1-D bulk copies
//    (cp.async.bulk) completing on mbarriers, issuing its first copies while
//    prep still runs; eight consumer warps each take 1/8 of a tile: the
//    partial sum of exp(x - R_b) on packed f32x2 FMAs and ex2, the maximum,
//    and the logits >= tau_b, appended to the beam's candidate list.  Nothing
//    in the loop waits on another CTA.
// 3. finish (one CTA per beam): lse_b from the partials, and the candidates'
//    scores histogrammed (upper 16 bits of an order-preserving key) into a
//    global histogram.  A beam whose threshold missed (too few or too many
//    candidates) is first redone exactly from its row.
// 4. final: every CTA reads from the histogram the bin B* that holds the
//    global 2W-th best score, the CTAs copy their beams' candidates in bins
//    >= B* to a small list, and the last CTA to finish sorts that list
//    (bitonic, in shared memory) with the full order and writes the 2W
//    results.  A list that would overflow (huge score ties) is resolved by an
//    exact radix select over all candidates instead.
//
// Every wait on an mbarrier is bounded; a wait that runs out marks the call
// failed and the outputs are filled with -1 ids and NaN scores.
#include <algorithm>
#include <cfloat>
#include <cstdint>
#include <mutex>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "slm_internal.h"
#include "sm103_ptx.cuh"

namespace slm {
namespace sel {

constexpr int kTile = 8192;                        // logits per streamed tile (16 KB)
constexpr int kCWarps = 8;                         // consumer warps of the stream kernel
constexpr int kVec = 4;                            // 16-byte vectors per lane and chunk
constexpr int kChunkElems = kVec * 8 * 32;         // 1024 logits per chunk
constexpr int kChunks = kTile / kChunkElems;       // 8 chunks per tile
constexpr int kStages = 12;                        // ring depth (192 KB)
constexpr int kSegCap = 256;                       // candidate slots per tile (rows longer than a tile)
constexpr int kStreamThreads = 32 * (kCWarps + 1);
constexpr int kCap = 8192;                         // candidates per beam
constexpr int kLocalBins = 1024;                   // per-beam score histogram in shared memory
constexpr int kMaxTiles = (1 << 24) / kTile;       // tiles per row at the largest vocabulary
constexpr int kFineBins = 65536;                   // global score histogram (key >> 16)
constexpr int kEliteMax = 4096;                    // entries the final ranking holds, at most
constexpr int kPrepThreads = 256;
constexpr int kSamples = 4096;
constexpr int kFinalThreads = 256;
constexpr int kFinalWarps = kFinalThreads / 32;
constexpr float kLog2e = 1.4426950408889634f;
static_assert(kCap >= kTile, "a one-tile row must fit the candidate list whole");
constexpr uint32_t kNegInf2 = 0xFF80FF80u;         // two bf16 -inf
constexpr unsigned kFull = 0xffffffffu;

// misc words of the workspace
constexpr int kMiscElite = 0;    // entries appended to the final list
constexpr int kMiscTicket = 1;   // final-kernel CTAs done
constexpr int kMiscMaxKey = 2;   // largest candidate score key
constexpr int kMiscStatus = 3;   // nonzero: a bounded wait ran out or the histogram was inconsistent

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

__device__ __forceinline__ float key_to_f32(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// Beam-local key: larger = earlier (higher logit, then lower id).
__device__ __forceinline__ unsigned long long local_key(uint32_t key16, uint32_t token) {
  return (static_cast<unsigned long long>(key16) << 32) | (0xFFFFFFFFu - token);
}

// A candidate as stored: bf16 bits in 32..47, token id in 0..31.
__device__ __forceinline__ unsigned long long cand_entry(uint32_t bits, uint32_t token) {
  return (static_cast<unsigned long long>(bits & 0xFFFFu) << 32) | token;
}

// Score key of a candidate of beam b: fl32(cum + fl32(x - lse)), order-preserving.
__device__ __forceinline__ uint32_t score_key(unsigned long long e, float cum, float lse) {
  const float x = bf16_bits_to_f32(static_cast<uint32_t>(e >> 32));
  return f32_key(__fadd_rn(cum, __fsub_rn(x, lse)));
}

// Global order as a 128-bit key (hi, lo), larger = earlier: score, then lower
// parent, then higher logit; lo = lower token id.
__device__ __forceinline__ ulonglong2 global_entry(uint32_t skey, uint32_t parent, unsigned long long e) {
  ulonglong2 g;
  g.x = (static_cast<unsigned long long>(skey) << 32) | ((0xFFFFu - parent) << 16) |
        bf16_key(static_cast<uint32_t>(e >> 32));
  g.y = 0xFFFFFFFFull - static_cast<uint32_t>(e);
  return g;
}

__device__ __forceinline__ bool entry_greater(const ulonglong2& a, const ulonglong2& b) {
  return a.x > b.x || (a.x == b.x && a.y > b.y);
}

// ---------------------------------------------------------------------------
// Small PTX helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// (d0, d1) = (a0 * b + c, a1 * b + c) in one packed f32x2 FMA.
__device__ __forceinline__ void fma2(float& d0, float& d1, float a0, float a1, float b, float c) {
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %4};\n\t"
      "mov.b64 rc, {%5, %5};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b), "f"(c));
}

// (s0, s1) += (e0, e1) in one packed f32x2 add (an FMA with unit factor).
__device__ __forceinline__ void add2(float& s0, float& s1, float e0, float e1) {
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %4};\n\t"
      "mov.b64 rc, {%0, %1};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "+f"(s0), "+f"(s1)
      : "f"(e0), "f"(e1), "f"(1.0f));
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void red_add(unsigned* p, unsigned v) {
  asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// 1-D bulk copy global -> shared, completing on an mbarrier; the source is
// read once, so it is marked first to leave L2.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* src, uint32_t bytes, uint64_t* bar,
                                          uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
          "r"(smem_u32(smem_dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// ---------------------------------------------------------------------------
// Warp reductions
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_max(float v) {
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

__device__ __forceinline__ uint32_t warp_max_u32(uint32_t v) {
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

__device__ __forceinline__ unsigned long long warp_min_u64(unsigned long long v) {
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

__device__ __forceinline__ int warp_inclusive_scan(int v, int lane) {
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += y;
  }
  return v;
}

// Finds in a 256-bin histogram (bins walked from 255 down) the bin holding
// the k-th largest item: its digit, the items above it, the items in it.
// Every lane of the warp calls it and gets the result.
__device__ __forceinline__ void warp_pick(const unsigned* hist, int k, int lane, int* digit, int* above,
                                          int* in_bin) {
  int local[8];
  int s = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    local[i] = static_cast<int>(hist[255 - 8 * lane - i]);
    s += local[i];
  }
  const int incl = warp_inclusive_scan(s, lane);
  const int excl = incl - s;
  const unsigned ball = __ballot_sync(kFull, excl < k && incl >= k);
  const int owner = ball ? (__ffs(ball) - 1) : 31;
  int d = 0, cum = 0, inb = 0;
  if (lane == owner) {
    cum = excl;
    d = 255 - 8 * lane - 7;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (cum + local[i] >= k) {
        d = 255 - 8 * lane - i;
        inb = local[i];
        break;
      }
      cum += local[i];
    }
  }
  *digit = __shfl_sync(kFull, d, owner);
  *above = __shfl_sync(kFull, cum, owner);
  *in_bin = __shfl_sync(kFull, inb, owner);
}

// ---------------------------------------------------------------------------
// Parameters
// ---------------------------------------------------------------------------
struct Params {
  const uint16_t* logits;  // [W_in, V] bf16 bits
  const float* cum;        // [W_in]
  int W_in, V, K, W;       // K = 2W candidates kept globally
  int n_tpr, n_tiles;      // tiles per row, tiles in all
  int seg_cap;             // candidate slots per tile
  bool vec_ok;             // rows 16-byte aligned: bulk copies and vector loads
  // workspace
  float* tau;                  // [W_in] candidate threshold
  float* ref;                  // [W_in] softmax reference R_b
  float* lse;                  // [W_in]
  int* cand_count;             // [W_in] entries of cand
  unsigned long long* seg;     // [W_in, n_tpr, seg_cap] candidates as the stream finds them
  float4* partial;             // [W_in, n_tpr] (reference, sum of exp, max logit, candidates as int bits)
  unsigned long long* cand;    // [W_in, kCap] each beam's candidates, contiguous
  unsigned* fine;              // [kFineBins]
  unsigned* misc;              // [4]
  ulonglong2* elite;           // [elite_cap]
  int elite_cap;
  // outputs
  int32_t* out_token;
  int32_t* out_parent;
  float* out_score;
  int32_t* out_cand_token;
  int32_t* out_cand_parent;
  float* out_cand_score;
  float* out_lse;
};

// ---------------------------------------------------------------------------
// 1. prep
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kPrepThreads) prep_kernel(const Params p) {
  grid_dep_launch();
  constexpr int kPerThread = kSamples / kPrepThreads;  // 16 sampled logits per thread
  static_assert(kPrepThreads == 256, "one histogram bin per thread");
  __shared__ unsigned hist[256];
  __shared__ unsigned wmaxk[kPrepThreads / 32];
  __shared__ int tau_key, found;
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, w = tid >> 5;

  if (b == 0 && tid < 4) p.misc[tid] = 0;
  {
    const int n4 = kFineBins / 4;
    const int per = (n4 + gridDim.x - 1) / gridDim.x;
    uint4* f4 = reinterpret_cast<uint4*>(p.fine);
    const int end = min(n4, (b + 1) * per);
    for (int i = b * per + tid; i < end; i += kPrepThreads) f4[i] = make_uint4(0u, 0u, 0u, 0u);
  }

  // 4096 sampled logits as order-preserving 16-bit keys
  const uint16_t* row = p.logits + static_cast<int64_t>(b) * p.V;
  uint32_t key[kPerThread];
  if (p.vec_ok) {
    // 512 runs of 8 logits (16 bytes) at evenly spaced, 8-aligned offsets
    constexpr int kRuns = kSamples / 8;
#pragma unroll
    for (int k = 0; k < kPerThread / 8; ++k) {
      const int j = tid + k * kPrepThreads;
      const int64_t off = (static_cast<int64_t>(j) * (p.V - 8) / (kRuns - 1)) & ~int64_t(7);
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(row + off));
      const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        key[8 * k + 2 * h] = bf16_key(wd[h] & 0xFFFFu);
        key[8 * k + 2 * h + 1] = bf16_key(wd[h] >> 16);
      }
    }
  } else {
#pragma unroll
    for (int k = 0; k < kPerThread; ++k) {
      const int s_ = tid + k * kPrepThreads;
      key[k] = bf16_key(row[static_cast<int64_t>(s_) * (p.V - 1) / (kSamples - 1)]);
    }
  }
  uint32_t mk = 0;
#pragma unroll
  for (int k = 0; k < kPerThread; ++k) mk = max(mk, key[k]);
  mk = warp_max_u32(mk);
  if (lane == 0) wmaxk[w] = mk;
  __syncthreads();
  uint32_t M = wmaxk[0];
  for (int i = 1; i < kPrepThreads / 32; ++i) M = max(M, wmaxk[i]);
  if (tid == 0) p.ref[b] = bf16_bits_to_f32(key_to_bf16(M));
  if (p.V <= kCap) {  // the whole row fits the candidate list
    if (tid == 0) p.tau[b] = -INFINITY;
    return;
  }
  // tau_b: the r-th largest sample, r a few standard deviations above the
  // expected sample count of the beam's K best.  The keys just below the
  // maximum are histogrammed (256 bins); a window too narrow to hold r
  // samples is widened 16-fold.
  const float expect = static_cast<float>(p.K) * kSamples / p.V;
  const int r = min(kSamples, static_cast<int>(ceilf(expect + 6.f * sqrtf(expect) + 8.f)));
  for (int sh = 0; sh <= 8; sh += 4) {
    hist[tid] = 0u;  // kPrepThreads == 256 bins
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kPerThread; ++k) {
      const uint32_t d = (M - key[k]) >> sh;
      if (d < 256u) atomicAdd(&hist[255u - d], 1u);
    }
    __syncthreads();
    if (w == 0) {
      int in_window = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) in_window += static_cast<int>(hist[8 * lane + i]);
      in_window = __shfl_sync(kFull, warp_inclusive_scan(in_window, lane), 31);
      int digit = 0, above, in_bin;
      if (in_window >= r) warp_pick(hist, r, lane, &digit, &above, &in_bin);
      // bin 255 - d holds the keys with (M - key) >> sh == d
      if (lane == 0) {
        found = (in_window >= r);
        tau_key = static_cast<int>(M) - ((255 - digit + 1) << sh) + 1;
      }
    }
    __syncthreads();
    if (found || sh == 8) break;
    __syncthreads();
  }
  if (tid == 0) {
    // keys below that of -inf (NaN patterns) clamp to -inf
    const uint32_t k = static_cast<uint32_t>(max(tau_key, static_cast<int>(bf16_key(0xFF80u))));
    p.tau[b] = bf16_bits_to_f32(key_to_bf16(k));
  }
}

// ---------------------------------------------------------------------------
// 2. stream
// ---------------------------------------------------------------------------
struct StreamSmem {
  uint4 ring[kStages][kTile / 8];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  int abort;
};

__device__ void stream_producer(const Params& p, StreamSmem& sh, int lane) {
  const uint64_t pol = evict_first_policy();
  int i = 0;
  for (int t = blockIdx.x; t < p.n_tiles; t += gridDim.x, ++i) {
    const int s = i % kStages;
    if (i >= kStages) {
      bool ok = mbar_wait(&sh.empty[s], ((i / kStages) - 1) & 1, &sh.abort);
      if (!__all_sync(kFull, ok)) break;
    }
    const int b = t / p.n_tpr, c = t - b * p.n_tpr;
    const int n = min(kTile, p.V - c * kTile);
    const uint16_t* src = p.logits + static_cast<int64_t>(b) * p.V + static_cast<int64_t>(c) * kTile;
    if (p.vec_ok) {
      if (lane == 0) {
        mbar_arrive_expect_tx(&sh.full[s], static_cast<uint32_t>(n) * 2u);
        bulk_load(&sh.ring[s][0], src, static_cast<uint32_t>(n) * 2u, &sh.full[s], pol);
      }
    } else {
      // unaligned rows: the warp copies the tile with 2-byte loads and pads
      // the last vector with -inf
      uint16_t* dst = reinterpret_cast<uint16_t*>(&sh.ring[s][0]);
      const int n8 = (n + 7) & ~7;
      for (int e = lane; e < n8; e += 32) dst[e] = (e < n) ? src[e] : static_cast<uint16_t>(0xFF80u);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.full[s]);
    }
  }
  // let the copies in flight land before the CTA can exit
  if (p.vec_ok && lane == 0) {
    for (int j = max(0, i - kStages); j < i; ++j) mbar_wait_drain(&sh.full[j % kStages], (j / kStages) & 1);
  }
}

// Sum over one chunk of exp(x - m), m = -cc / log2(e), on packed f32x2.
__device__ __forceinline__ void chunk_exp_sum(const uint4 (&r)[kVec], float cc, float& s0, float& s1, float& s2,
                                              float& s3) {
#pragma unroll
  for (int v = 0; v < kVec; ++v) {
    const uint32_t wd[4] = {r[v].x, r[v].y, r[v].z, r[v].w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      float y0, y1;
      fma2(y0, y1, __uint_as_float(wd[h] << 16), __uint_as_float(wd[h] & 0xFFFF0000u), kLog2e, cc);
      if (h & 1) add2(s2, s3, ex2(y0), ex2(y1));
      else add2(s0, s1, ex2(y0), ex2(y1));
    }
  }
}

// Loads chunk ch of a ring slot: vector v of the lane holds tile logits
// (ch * 1024 + (v * 32 + lane) * 8) + 0..7; vectors past the tile's n logits
// read as -inf.
__device__ __forceinline__ void load_chunk(const uint4* slot, int ch, int lane, int n, uint4 (&r)[kVec]) {
#pragma unroll
  for (int v = 0; v < kVec; ++v) {
    const int e0 = ch * kChunkElems + (v * 32 + lane) * 8;
    r[v] = (e0 < n) ? slot[ch * (kChunkElems / 8) + v * 32 + lane]
                    : make_uint4(kNegInf2, kNegInf2, kNegInf2, kNegInf2);
  }
}

// Consumer warp cw takes the CTA's tiles cw, cw + 8, cw + 16, ... whole, so
// the warps work on different tiles and no warp waits for another.  Per
// chunk of 1024 logits a lane holds 32: it adds their exp(x - R_b) to its
// sums and marks those >= tau_b in a 32-bit mask (bit 4v + h for the low
// logit of word h of vector v, bit 16 + 4v + h for the high one).  After the
// tile one warp scan places the marked logits in the tile's candidate
// segment; they are read back from the ring slot, which is released only then.
__device__ void stream_consumer(const Params& p, StreamSmem& sh, int cw, int lane) {
  grid_dep_wait();  // tau, ref and the reset counters come from the prep kernel
  const int step = kCWarps * gridDim.x;
  int t = blockIdx.x + cw * gridDim.x;
  float tau_n = 0.f, ref_n = 0.f;
  if (t < p.n_tiles) {
    tau_n = __ldcg(p.tau + t / p.n_tpr);
    ref_n = __ldcg(p.ref + t / p.n_tpr);
  }
  for (int i = cw; t < p.n_tiles; i += kCWarps, t += step) {
    const int s = i % kStages;
    const int b = t / p.n_tpr, c = t - b * p.n_tpr;
    const int n = min(kTile, p.V - c * kTile);
    const float tau = tau_n, R0 = ref_n;
    if (t + step < p.n_tiles) {  // the next tile's beam values, early
      tau_n = __ldcg(p.tau + (t + step) / p.n_tpr);
      ref_n = __ldcg(p.ref + (t + step) / p.n_tpr);
    }
    const bool ok = mbar_wait(&sh.full[s], (i / kStages) & 1, &sh.abort);
    if (!__all_sync(kFull, ok)) break;

    const uint4* slot = &sh.ring[s][0];
    const bool keep_all = !(tau > -INFINITY);  // rows of one tile: every logit is a candidate
    const __nv_bfloat162 t2 = __float2bfloat162_rn(tau);  // tau is a bf16 value or -inf
    const float mref = (R0 > -INFINITY) ? R0 : 0.f;
    const float cc = -mref * kLog2e;
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
    uint32_t cb[kChunks];
#pragma unroll
    for (int ch = 0; ch < kChunks; ++ch) {
      uint4 r[kVec];
      load_chunk(slot, ch, lane, n, r);
      chunk_exp_sum(r, cc, s0, s1, s2, s3);
      uint32_t bits = 0u;
#pragma unroll
      for (int v = 0; v < kVec; ++v) {
        const uint32_t wd[4] = {r[v].x, r[v].y, r[v].z, r[v].w};
#pragma unroll
        for (int h = 0; h < 4; ++h)
          bits |= __hge2_mask(*reinterpret_cast<const __nv_bfloat162*>(&wd[h]), t2) & (0x00010001u << (4 * v + h));
      }
      if (keep_all) {  // -inf padding past the tile's end must not count
#pragma unroll
        for (int v = 0; v < kVec; ++v) {
          const int nv = min(max(n - (ch * kChunkElems + (v * 32 + lane) * 8), 0), 8);
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            if (2 * h >= nv) bits &= ~(1u << (4 * v + h));
            if (2 * h + 1 >= nv) bits &= ~(1u << (16 + 4 * v + h));
          }
        }
      }
      cb[ch] = bits;
    }

    // candidates to the tile's segment, in lane order
    int cnt = 0;
#pragma unroll
    for (int ch = 0; ch < kChunks; ++ch) cnt += __popc(cb[ch]);
    const int incl = warp_inclusive_scan(cnt, lane);
    const int found = __shfl_sync(kFull, incl, 31);
    int pos = incl - cnt;
    unsigned long long* seg = p.seg + (static_cast<int64_t>(b) * p.n_tpr + c) * p.seg_cap;
    const uint16_t* slot16 = reinterpret_cast<const uint16_t*>(slot);
    float cmax = -INFINITY;  // largest candidate of the lane
#pragma unroll
    for (int ch = 0; ch < kChunks; ++ch) {
      uint32_t bits = cb[ch];
      while (bits) {
        const int j = __ffs(bits) - 1;
        bits &= bits - 1u;
        const int q = j & 15;
        const int e = ch * kChunkElems + ((q >> 2) * 32 + lane) * 8 + 2 * (q & 3) + (j >> 4);
        const uint32_t xb = slot16[e];
        cmax = fmaxf(cmax, bf16_bits_to_f32(xb));
        if (pos < p.seg_cap) seg[pos] = cand_entry(xb, static_cast<uint32_t>(c * kTile + e));
        ++pos;
      }
    }
    // A candidate far above the reference (possible only when the sample
    // missed the row's top) overflowed exp: this lane's sum is redone against
    // its own maximum.
    float m_l = mref;
    if (cmax - mref > 64.f) {
      m_l = cmax;
      s0 = s1 = s2 = s3 = 0.f;
#pragma unroll 1
      for (int ch = 0; ch < kChunks; ++ch) {
        uint4 r[kVec];
        load_chunk(slot, ch, lane, n, r);
        chunk_exp_sum(r, -m_l * kLog2e, s0, s1, s2, s3);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.empty[s]);  // the slot's data is no longer read

    // the tile's partial: common reference, sum, largest candidate, count
    const float M = warp_max(m_l);
    float l = (s0 + s1) + (s2 + s3);
    if (m_l != M) l *= ex2((m_l - M) * kLog2e);
    l = warp_sum(l);
    const float wm = warp_max(cmax);
    if (lane == 0) p.partial[static_cast<int64_t>(b) * p.n_tpr + c] = make_float4(M, l, wm, __int_as_float(found));
  }
}

__global__ void __launch_bounds__(kStreamThreads, 1) stream_kernel(const Params p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  StreamSmem& sh = *reinterpret_cast<StreamSmem*>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], 1);
    }
    sh.abort = 0;
    fence_mbarrier_init();
  }
  __syncthreads();
  grid_dep_launch();
  if (warp == 0) stream_producer(p, sh, lane);
  else stream_consumer(p, sh, warp - 1, lane);
  __syncthreads();
  if (threadIdx.x == 0 && sh.abort) atomicOr(p.misc + kMiscStatus, 1u);
}

// ---------------------------------------------------------------------------
// Block primitives of the finish and final kernels (kBlockThreads threads)
// ---------------------------------------------------------------------------
struct Scratch {
  unsigned whist[kFinalWarps][256];
  unsigned hist[256];
  unsigned lbins[kLocalBins];
  unsigned long long wu64[2][kFinalWarps];
  float wf[kFinalWarps];
  int wint[kFinalWarps];
  int digit, above, in_bin, counter, flag, bstar, bstar_above, bstar_count;
  unsigned long long u64;
};

__device__ __forceinline__ float block_max(float v, Scratch& sh) {
  v = warp_max(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sh.wf[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = sh.wf[0];
  for (int i = 1; i < kFinalWarps; ++i) r = fmaxf(r, sh.wf[i]);
  return r;
}

__device__ __forceinline__ uint32_t block_max_u32(uint32_t v, Scratch& sh) {
  v = warp_max_u32(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sh.wint[threadIdx.x >> 5] = static_cast<int>(v);
  __syncthreads();
  uint32_t r = 0;
  for (int i = 0; i < kFinalWarps; ++i) r = max(r, static_cast<uint32_t>(sh.wint[i]));
  return r;
}

// Sum in a fixed order (deterministic).
__device__ __forceinline__ float block_sum(float v, Scratch& sh) {
  v = warp_sum(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sh.wf[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = 0.f;
  for (int i = 0; i < kFinalWarps; ++i) r += sh.wf[i];
  return r;
}

__device__ __forceinline__ int block_scan_excl(int v, int* total, Scratch& sh) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int x = warp_inclusive_scan(v, lane);
  __syncthreads();
  if (lane == 31) sh.wint[w] = x;
  __syncthreads();
  int base = 0, tot = 0;
  for (int i = 0; i < kFinalWarps; ++i) {
    if (i < w) base += sh.wint[i];
    tot += sh.wint[i];
  }
  *total = tot;
  return base + x - v;
}

// k-th largest (1-based, counting repeats) of the 64-bit keys all threads
// visit with for_each(f).  Each pass histograms the keys in the live range
// [lo, hi] by the 8 bits below the range's leading bit and narrows the range
// to the bin holding the k-th key; a bin with a single key ends it.
template <class ForEach>
__device__ unsigned long long block_kth(ForEach for_each, int k, Scratch& sh) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  unsigned long long lo = ~0ull, hi = 0ull;
  for_each([&](unsigned long long key) {
    lo = min(lo, key);
    hi = max(hi, key);
  });
  lo = warp_min_u64(lo);
  hi = warp_max_u64(hi);
  __syncthreads();
  if (lane == 0) {
    sh.wu64[0][w] = lo;
    sh.wu64[1][w] = hi;
  }
  __syncthreads();
  lo = ~0ull;
  hi = 0ull;
  for (int i = 0; i < kFinalWarps; ++i) {
    lo = min(lo, sh.wu64[0][i]);
    hi = max(hi, sh.wu64[1][i]);
  }
  while (lo < hi) {
    const int sft = max(0, 64 - __clzll(hi - lo) - 8);
    for (int i = threadIdx.x; i < kFinalWarps * 256; i += kFinalThreads) (&sh.whist[0][0])[i] = 0u;
    __syncthreads();
    const unsigned long long lo_c = lo, hi_c = hi;
    for_each([&](unsigned long long key) {
      if (key >= lo_c && key <= hi_c) atomicAdd(&sh.whist[w][static_cast<uint32_t>((key - lo_c) >> sft)], 1u);
    });
    __syncthreads();
    {
      unsigned s = 0;
      for (int i = 0; i < kFinalWarps; ++i) s += sh.whist[i][threadIdx.x];  // kFinalThreads == 256
      sh.hist[threadIdx.x] = s;
    }
    __syncthreads();
    if (w == 0) {
      int digit, above, in_bin;
      warp_pick(sh.hist, k, lane, &digit, &above, &in_bin);
      if (lane == 0) {
        sh.digit = digit;
        sh.above = above;
        sh.in_bin = in_bin;
      }
    }
    __syncthreads();
    const unsigned long long base = lo + (static_cast<unsigned long long>(sh.digit) << sft);
    const unsigned long long width = (1ull << sft) - 1;
    hi = (hi - base <= width) ? hi : base + width;
    lo = base;
    k -= sh.above;
    const int in_bin = sh.in_bin;
    __syncthreads();
    if (in_bin == 1 && lo < hi) {
      const unsigned long long lo_b = lo, hi_b = hi;
      for_each([&](unsigned long long key) {
        if (key >= lo_b && key <= hi_b) sh.u64 = key;
      });
      __syncthreads();
      const unsigned long long found = sh.u64;
      __syncthreads();
      return found;
    }
  }
  return lo;
}

// Descending bitonic sort of ent[0, n_pow2).
__device__ void block_sort_desc(ulonglong2* ent, int n_pow2) {
  for (int size = 2; size <= n_pow2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      __syncthreads();
      for (int t = threadIdx.x; t < n_pow2 / 2; t += kFinalThreads) {
        const int lo = 2 * t - (t & (stride - 1));
        const int hi = lo + stride;
        const bool desc = ((lo & size) == 0);
        const ulonglong2 a = ent[lo], b = ent[hi];
        if (entry_greater(b, a) == desc) {
          ent[lo] = b;
          ent[hi] = a;
        }
      }
    }
  }
  __syncthreads();
}

__device__ __forceinline__ int next_pow2(int x) {
  int q = 1;
  while (q < x) q <<= 1;
  return q;
}

// ---------------------------------------------------------------------------
// 3. finish (one CTA per beam)
// ---------------------------------------------------------------------------
// The threshold missed for beam b (too few logits above it, or more than the
// list holds): the beam's exact top K from its whole row replaces the list.
__device__ void exact_beam(const Params& p, Scratch& sh, int b) {
  const uint16_t* row = p.logits + static_cast<int64_t>(b) * p.V;
  const int V = p.V;
  auto for_each = [&](auto f) {
    for (int j = threadIdx.x; j < V; j += kFinalThreads) f(local_key(bf16_key(row[j]), static_cast<uint32_t>(j)));
  };
  const unsigned long long kth = block_kth(for_each, p.K, sh);
  if (threadIdx.x == 0) sh.counter = 0;
  __syncthreads();
  unsigned long long* dst = p.cand + static_cast<int64_t>(b) * kCap;
  for (int j = threadIdx.x; j < V; j += kFinalThreads) {
    const uint32_t bits = row[j];
    if (local_key(bf16_key(bits), static_cast<uint32_t>(j)) >= kth) {
      const int pos = atomicAdd(&sh.counter, 1);
      if (pos < kCap) dst[pos] = cand_entry(bits, static_cast<uint32_t>(j));
    }
  }
  __threadfence();  // the list is read back below from L2
  __syncthreads();
  if (threadIdx.x == 0) p.cand_count[b] = p.K;
}

// Beam b: lse_b from the stream partials; the tiles' candidate segments
// gathered into one list; the candidates' scores into the global histogram
// and the largest score key into misc.
//
// Rows of up to 32 tiles (vocabularies up to 262,144) take a path without
// block-wide steps before the histogram: every warp reads all of the beam's
// partials (lse_b and the segment offsets come out of warp reductions, the
// same in every warp), finds the tile of each list entry it moves by a
// binary search over the lanes, and requests eight entries per thread at once.
constexpr int kFastTiles = 32;

__global__ void __launch_bounds__(kFinalThreads) finish_kernel(const Params p) {
  __shared__ Scratch sh;
  __shared__ int start[kMaxTiles + 1];  // first list entry of each tile's segment
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
  uint32_t kmax = 0;  // largest score key this thread histograms
  for (int d = tid; d < kLocalBins; d += kFinalThreads) sh.lbins[d] = 0u;
  __syncthreads();
  grid_dep_wait();
  grid_dep_launch();
  const int nt = p.n_tpr;
  const float4* P = p.partial + static_cast<int64_t>(b) * nt;
  const unsigned long long* seg = p.seg + static_cast<int64_t>(b) * nt * p.seg_cap;
  unsigned long long* cand = p.cand + static_cast<int64_t>(b) * kCap;
  const float cum = __ldg(p.cum + b);

  float lse, top;
  int count;
  bool over;
  if (nt <= kFastTiles) {
    const float4 q = (lane < nt) ? __ldcg(P + lane) : make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
    const float M = warp_max(q.y > 0.f ? q.x : -INFINITY);
    top = warp_max(q.z);
    const float L = warp_sum(q.y > 0.f ? q.y * ex2((q.x - M) * kLog2e) : 0.f);
    lse = M + logf(L);
    const int cnt = (lane < nt) ? __float_as_int(q.w) : 0;
    over = __any_sync(kFull, cnt > p.seg_cap);
    const int incl = warp_inclusive_scan(cnt, lane);
    const int st = incl - cnt;  // lane j: first list entry of tile j
    count = __shfl_sync(kFull, incl, 31);
    if (!(over || count < p.K || count > kCap)) {
      const uint32_t top_bin = f32_key(__fadd_rn(cum, __fsub_rn(top, lse))) >> 16;
      for (int e0 = 0; e0 < count; e0 += 8 * kFinalThreads) {
        unsigned long long v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int e = e0 + k * kFinalThreads + tid;
          // the tile holding entry e: the last j with start_j <= e
          int j = 0;
#pragma unroll
          for (int stp = 16; stp > 0; stp >>= 1) {
            const int s_j = __shfl_sync(kFull, st, j + stp);
            if (j + stp < nt && s_j <= e) j += stp;
          }
          const int sj = __shfl_sync(kFull, st, j);
          v[k] = (e < count) ? __ldcg(seg + static_cast<int64_t>(j) * p.seg_cap + (e - sj)) : 0ull;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int e = e0 + k * kFinalThreads + tid;
          if (e < count) {
            cand[e] = v[k];
            const uint32_t sk = score_key(v[k], cum, lse);
            kmax = max(kmax, sk);
            const uint32_t bin = sk >> 16;
            const uint32_t d = top_bin - bin;
            if (d < static_cast<uint32_t>(kLocalBins)) atomicAdd(&sh.lbins[d], 1u);
            else red_add(p.fine + bin, 1u);
          }
        }
      }
    }
  } else {
    float M = -INFINITY;
    top = -INFINITY;
    over = false;
    for (int j = tid; j < nt; j += kFinalThreads) {
      const float4 q = __ldcg(P + j);
      if (q.y > 0.f) M = fmaxf(M, q.x);
      top = fmaxf(top, q.z);
      over |= __float_as_int(q.w) > p.seg_cap;
    }
    M = block_max(M, sh);
    top = block_max(top, sh);
    over = __syncthreads_or(over);
    float L = 0.f;
    for (int j = tid; j < nt; j += kFinalThreads) {
      const float4 q = __ldcg(P + j);
      if (q.y > 0.f) L += q.y * ex2((q.x - M) * kLog2e);
    }
    L = block_sum(L, sh);
    lse = M + logf(L);
    // segment starts (exclusive prefix of the tiles' counts)
    int carry = 0;
    for (int j0 = 0; j0 < nt; j0 += kFinalThreads) {
      const int j = j0 + tid;
      const int cj = (j < nt) ? __float_as_int(__ldcg(&P[j].w)) : 0;
      int tot;
      const int ex = block_scan_excl(cj, &tot, sh);
      if (j < nt) start[j] = carry + ex;
      carry += tot;
    }
    if (tid == 0) start[nt] = carry;
    __syncthreads();
    count = carry;
    if (!(over || count < p.K || count > kCap)) {
      const uint32_t top_bin = f32_key(__fadd_rn(cum, __fsub_rn(top, lse))) >> 16;
      for (int e = tid; e < count; e += kFinalThreads) {
        int lo = 0, hi = nt - 1;  // the tile whose segment holds entry e
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (start[mid] <= e) lo = mid;
          else hi = mid - 1;
        }
        const unsigned long long entry = __ldcg(seg + static_cast<int64_t>(lo) * p.seg_cap + (e - start[lo]));
        cand[e] = entry;
        const uint32_t sk = score_key(entry, cum, lse);
        kmax = max(kmax, sk);
        const uint32_t bin = sk >> 16;
        const uint32_t d = top_bin - bin;
        if (d < static_cast<uint32_t>(kLocalBins)) atomicAdd(&sh.lbins[d], 1u);
        else red_add(p.fine + bin, 1u);
      }
    }
  }
  if (tid == 0) {
    p.lse[b] = lse;
    if (p.out_lse) p.out_lse[b] = lse;
  }
  // the row maximum is a candidate, so its score is the beam's largest
  uint32_t top_bin = f32_key(__fadd_rn(cum, __fsub_rn(top, lse))) >> 16;
  if (over || count < p.K || count > kCap) {
    // the threshold missed: the exact top K from the whole row
    exact_beam(p, sh, b);
    count = p.K;
    for (int i = tid; i < count; i += kFinalThreads) kmax = max(kmax, score_key(__ldcg(cand + i), cum, lse));
    // the window starts at the largest key of the exact list itself
    const uint32_t kb = block_max_u32(kmax, sh);
    top_bin = kb >> 16;
    for (int i = tid; i < count; i += kFinalThreads) {
      const uint32_t sk = score_key(__ldcg(cand + i), cum, lse);
      kmax = max(kmax, sk);
      const uint32_t bin = sk >> 16;
      const uint32_t d = top_bin - bin;
      if (d < static_cast<uint32_t>(kLocalBins)) atomicAdd(&sh.lbins[d], 1u);
      else red_add(p.fine + bin, 1u);
    }
  } else if (tid == 0) {
    p.cand_count[b] = count;
  }
  __syncthreads();
  for (int d = tid; d < kLocalBins; d += kFinalThreads) {
    const unsigned v = sh.lbins[d];
    if (v) red_add(p.fine + (top_bin - d), v);
  }
  // the global walk starts at the largest key actually histogrammed (with
  // finite logits that of the row maximum; it also bounds NaN-derived keys)
  kmax = warp_max_u32(kmax);
  if (lane == 0) atomicMax(p.misc + kMiscMaxKey, kmax);
}

// ---------------------------------------------------------------------------
// 4. final
// ---------------------------------------------------------------------------
constexpr int kRankBins = 1024;  // score bins the final ranking spans without a full sort

// Dynamic shared memory of the final kernel: this head, then elite_cap
// entries (as ulonglong2, or as separate hi / lo arrays for the ranking).
struct FinalHead {
  Scratch sc;
  int pre[kRankBins];   // entries of the list in bins above bin S - d
  int fill[kRankBins];  // entries placed so far in bin S - d
};

// Result r of the global order; error = true writes -1 ids and NaN scores.
__device__ __forceinline__ void write_result(const Params& p, int r, const ulonglong2& g, bool error = false) {
  const int token = error ? -1 : static_cast<int>(0xFFFFFFFFull - g.y);
  const int parent = error ? -1 : 0xFFFF - static_cast<int>((g.x >> 16) & 0xFFFFull);
  const float score = error ? __int_as_float(0x7fc00000) : key_to_f32(static_cast<uint32_t>(g.x >> 32));
  if (r < p.W) {
    p.out_token[r] = token;
    p.out_parent[r] = parent;
    p.out_score[r] = score;
  }
  if (p.out_cand_token) p.out_cand_token[r] = token;
  if (p.out_cand_parent) p.out_cand_parent[r] = parent;
  if (p.out_cand_score) p.out_cand_score[r] = score;
}

__global__ void __launch_bounds__(kFinalThreads, 1) final_kernel(const Params p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  FinalHead& fs = *reinterpret_cast<FinalHead*>(smem_raw);
  Scratch& sh = fs.sc;
  ulonglong2* ent = reinterpret_cast<ulonglong2*>(smem_raw + sizeof(FinalHead));
  const int cap = p.elite_cap;
  const int tid = threadIdx.x, lane = tid & 31;
  const int K = p.K;
  const int b = blockIdx.x;
  grid_dep_wait();

  // everything this CTA reads, requested at once: its beam's values, the
  // first candidates (the list buffer is always that long), the top key
  constexpr int kBatch = 8;
  const unsigned long long* cand = p.cand + static_cast<int64_t>(b) * kCap;
  unsigned long long e[kBatch];
#pragma unroll
  for (int k = 0; k < kBatch; ++k) e[k] = __ldcg(cand + k * kFinalThreads + tid);
  const int count = min(__ldcg(p.cand_count + b), kCap);
  const float lse = __ldcg(p.lse + b), cum = __ldg(p.cum + b);
  const int S = static_cast<int>(__ldcg(p.misc + kMiscMaxKey) >> 16);

  // B*: walking the histogram down from the largest score, the bin where the
  // running count first reaches K.  pre[] keeps the running counts of the
  // bins walked (for the ranking by the last CTA).
  {
    int top = S, carry = 0;
    if (tid == 0) sh.bstar = -1;
    while (true) {
      const int bin = top - tid;
      const int c = (bin >= 0) ? static_cast<int>(__ldcg(p.fine + bin)) : 0;
      int total;
      const int excl = block_scan_excl(c, &total, sh);
      if (S - bin < kRankBins) fs.pre[S - bin] = carry + excl;
      if (carry + excl < K && carry + excl + c >= K) {
        sh.bstar = bin;
        sh.bstar_above = carry + excl;
        sh.bstar_count = c;
      }
      carry += total;
      if (carry >= K || top - kFinalThreads < 0) break;
      top -= kFinalThreads;
    }
    __syncthreads();
  }
  const int bstar = sh.bstar;
  if (bstar < 0 && tid == 0) atomicOr(p.misc + kMiscStatus, 2u);

  // this beam's candidates in bins >= B* to the final list
  if (bstar >= 0) {
    for (int i0 = 0; i0 < count; i0 += kBatch * kFinalThreads) {
      if (i0 > 0) {
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
          const int i = i0 + k * kFinalThreads + tid;
          e[k] = (i < count) ? __ldcg(cand + i) : 0ull;
        }
      }
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        if (i0 + k * kFinalThreads >= count) break;  // uniform across the CTA
        const int i = i0 + k * kFinalThreads + tid;
        bool take = false;
        ulonglong2 g = make_ulonglong2(0ull, 0ull);
        if (i < count) {
          const uint32_t sk = score_key(e[k], cum, lse);
          if (static_cast<int>(sk >> 16) >= bstar) {
            take = true;
            g = global_entry(sk, static_cast<uint32_t>(b), e[k]);
          }
        }
        const unsigned bal = __ballot_sync(kFull, take);
        if (bal) {
          unsigned base = 0;
          if (lane == 0) base = atomicAdd(p.misc + kMiscElite, static_cast<unsigned>(__popc(bal)));
          base = __shfl_sync(kFull, base, 0);
          const unsigned pos = base + __popc(bal & ((1u << lane) - 1u));
          if (take && pos < static_cast<unsigned>(cap)) p.elite[pos] = g;
        }
      }
    }
  }

  // the last CTA to finish ranks the list
  __syncthreads();
  if (tid == 0) sh.flag = (atom_add_acq_rel(p.misc + kMiscTicket, 1u) == gridDim.x - 1);
  __syncthreads();
  if (!sh.flag) return;

  const unsigned status = __ldcg(p.misc + kMiscStatus);
  const int n_e = static_cast<int>(__ldcg(p.misc + kMiscElite));
  // the list holds exactly the histogram's entries in bins >= B*
  if (status != 0u || bstar < 0 || n_e < K || n_e != sh.bstar_above + sh.bstar_count) {
    for (int r = tid; r < K; r += kFinalThreads) write_result(p, r, make_ulonglong2(0ull, 0ull), true);
    return;
  }

  if (n_e <= cap && S - bstar < kRankBins) {
    // Rank by bin: an entry's place is the count of the bins above its own
    // plus its rank among the (few) entries of its bin.  Entries are first
    // grouped by bin, then each compares itself with its group.
    unsigned long long* ehi = reinterpret_cast<unsigned long long*>(ent);
    uint32_t* elo = reinterpret_cast<uint32_t*>(ehi + cap);
    for (int d = tid; d <= S - bstar; d += kFinalThreads) fs.fill[d] = 0;
    if (tid == 0) sh.counter = 0;  // entries outside [B*, S]: none unless the histogram is inconsistent
    __syncthreads();
    for (int i = tid; i < n_e; i += kFinalThreads) {
      const unsigned long long hi = __ldcg(&p.elite[i].x);
      const uint32_t lo = static_cast<uint32_t>(__ldcg(&p.elite[i].y));
      const int d = S - static_cast<int>(hi >> 48);
      if (d < 0 || d > S - bstar) {
        atomicAdd(&sh.counter, 1);
        continue;
      }
      const int idx = fs.pre[d] + atomicAdd(&fs.fill[d], 1);
      if (idx < cap) {
        ehi[idx] = hi;
        elo[idx] = lo;
      }
    }
    __syncthreads();
    if (sh.counter != 0) {
      for (int r = tid; r < K; r += kFinalThreads) write_result(p, r, make_ulonglong2(0ull, 0ull), true);
      return;
    }
    for (int i = tid; i < n_e; i += kFinalThreads) {
      const unsigned long long hi = ehi[i];
      const uint32_t lo = elo[i];
      const int d = S - static_cast<int>(hi >> 48);
      const int g0 = fs.pre[d], gn = fs.fill[d];
      int rank = g0;
      const int g1 = min(g0 + gn, n_e);
#pragma unroll 4
      for (int j = g0; j < g1; ++j) {
        const unsigned long long hj = ehi[j];
        rank += (hj > hi) | ((hj == hi) & (elo[j] > lo));
      }
      if (rank < K) write_result(p, rank, make_ulonglong2(hi, lo));
    }
    return;
  }

  int n_sort;
  if (n_e <= cap) {
    n_sort = n_e;
    for (int i = tid; i < n_e; i += kFinalThreads) {
      ulonglong2 g;
      g.x = __ldcg(&p.elite[i].x);
      g.y = __ldcg(&p.elite[i].y);
      ent[i] = g;
    }
  } else {
    // Huge score ties: exact selection over every candidate in bins >= B*.
    auto for_each_entry = [&](auto f) {
      for (int bb = 0; bb < p.W_in; ++bb) {
        const int cnt = min(__ldcg(p.cand_count + bb), kCap);
        const float lse_b = __ldcg(p.lse + bb), cum_b = __ldg(p.cum + bb);
        const unsigned long long* cd = p.cand + static_cast<int64_t>(bb) * kCap;
        for (int i = tid; i < cnt; i += kFinalThreads) {
          const unsigned long long en = __ldcg(cd + i);
          const uint32_t sk = score_key(en, cum_b, lse_b);
          if (static_cast<int>(sk >> 16) >= bstar) f(global_entry(sk, static_cast<uint32_t>(bb), en));
        }
      }
    };
    const unsigned long long kth_hi =
        block_kth([&](auto f) { for_each_entry([&](const ulonglong2& g) { f(g.x); }); }, K, sh);
    int mine = 0;
    for_each_entry([&](const ulonglong2& g) { mine += (g.x > kth_hi); });
    int above;
    block_scan_excl(mine, &above, sh);
    const unsigned long long kth_lo = block_kth(
        [&](auto f) {
          for_each_entry([&](const ulonglong2& g) {
            if (g.x == kth_hi) f(g.y);
          });
        },
        K - above, sh);
    if (tid == 0) sh.counter = 0;
    __syncthreads();
    for_each_entry([&](const ulonglong2& g) {
      if (g.x > kth_hi || (g.x == kth_hi && g.y >= kth_lo)) {
        const int pos = atomicAdd(&sh.counter, 1);
        if (pos < cap) ent[pos] = g;
      }
    });
    __syncthreads();
    n_sort = K;
  }
  const int n2 = next_pow2(max(n_sort, 2));
  for (int i = n_sort + tid; i < n2; i += kFinalThreads) ent[i] = make_ulonglong2(0ull, 0ull);
  block_sort_desc(ent, n2);
  for (int r = tid; r < K; r += kFinalThreads) write_result(p, r, ent[r]);
}

}  // namespace sel

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
namespace {

struct SelLayout {
  int n_tpr, seg_cap, elite_cap;
  size_t off_tau, off_ref, off_lse, off_count, off_seg, off_partial, off_cand, off_fine, off_misc, off_elite, total;
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

bool sel_layout(int W_in, int V, int W, SelLayout* L) {
  if (W_in <= 0 || V <= 0 || W <= 0) return false;
  const int64_t K = 2 * static_cast<int64_t>(W);
  if (K > 2048 || K > V || W_in > 1024 || V >= (1 << 24)) return false;
  L->n_tpr = (V + sel::kTile - 1) / sel::kTile;
  // a row of one tile keeps every logit (tau = -inf)
  L->seg_cap = (L->n_tpr == 1) ? ((V + 7) & ~7) : sel::kSegCap;
  size_t o = 0;
  L->off_tau = o;     o = align256(o + sizeof(float) * size_t(W_in));
  L->off_ref = o;     o = align256(o + sizeof(float) * size_t(W_in));
  L->off_lse = o;     o = align256(o + sizeof(float) * size_t(W_in));
  L->off_count = o;   o = align256(o + sizeof(int) * size_t(W_in));
  L->off_seg = o;     o = align256(o + sizeof(unsigned long long) * size_t(W_in) * L->n_tpr * L->seg_cap);
  L->off_partial = o; o = align256(o + sizeof(float4) * size_t(W_in) * L->n_tpr);
  L->off_cand = o;    o = align256(o + sizeof(unsigned long long) * size_t(W_in) * sel::kCap);
  L->off_fine = o;    o = align256(o + sizeof(unsigned) * size_t(sel::kFineBins));
  L->off_misc = o;    o = align256(o + sizeof(unsigned) * 4);
  // the final list: 2K entries and room for a few ties, a power of two
  int cap = 512;
  while (cap < 2 * K && cap < sel::kEliteMax) cap <<= 1;
  L->elite_cap = cap;
  L->off_elite = o;   o = align256(o + sizeof(ulonglong2) * size_t(cap));
  L->total = o;
  return true;
}

int sm_count() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  std::lock_guard<std::mutex> lock(mu);
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

// Launches a kernel that may start while the previous kernel on the stream is
// still running; it waits for that kernel's results with griddepcontrol.wait.
template <class Kernel>
cudaError_t launch_dependent(Kernel kernel, int grid, int block, size_t smem, cudaStream_t stream,
                             const sel::Params& p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
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
  p.n_tpr = L.n_tpr;
  p.n_tiles = W_in * L.n_tpr;
  p.seg_cap = L.seg_cap;
  p.elite_cap = L.elite_cap;
  p.vec_ok = (V % 8 == 0) && ((reinterpret_cast<uintptr_t>(logits) & 15) == 0);
  p.tau = reinterpret_cast<float*>(ws + L.off_tau);
  p.ref = reinterpret_cast<float*>(ws + L.off_ref);
  p.lse = reinterpret_cast<float*>(ws + L.off_lse);
  p.cand_count = reinterpret_cast<int*>(ws + L.off_count);
  p.cand = reinterpret_cast<unsigned long long*>(ws + L.off_cand);
  p.seg = reinterpret_cast<unsigned long long*>(ws + L.off_seg);
  p.partial = reinterpret_cast<float4*>(ws + L.off_partial);
  p.fine = reinterpret_cast<unsigned*>(ws + L.off_fine);
  p.misc = reinterpret_cast<unsigned*>(ws + L.off_misc);
  p.elite = reinterpret_cast<ulonglong2*>(ws + L.off_elite);
  p.out_token = out_token;
  p.out_parent = out_parent;
  p.out_score = out_score;
  p.out_cand_token = out_cand_token;
  p.out_cand_parent = out_cand_parent;
  p.out_cand_score = out_cand_score;
  p.out_lse = out_lse;

  sel::prep_kernel<<<W_in, sel::kPrepThreads, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  const size_t smem_stream = sizeof(sel::StreamSmem);
  e = cudaFuncSetAttribute(sel::stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem_stream));
  if (e != cudaSuccess) return e;
  const int grid_stream = std::min(sm_count(), p.n_tiles);
  e = launch_dependent(sel::stream_kernel, grid_stream, sel::kStreamThreads, smem_stream, stream, p);
  if (e != cudaSuccess) return e;

  e = launch_dependent(sel::finish_kernel, W_in, sel::kFinalThreads, 0, stream, p);
  if (e != cudaSuccess) return e;

  const size_t smem_final = sizeof(sel::FinalHead) + sizeof(ulonglong2) * size_t(L.elite_cap);
  e = cudaFuncSetAttribute(sel::final_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem_final));
  if (e != cudaSuccess) return e;
  const int grid_final = W_in;
  return launch_dependent(sel::final_kernel, grid_final, sel::kFinalThreads, smem_final, stream, p);
}

}  // namespace slm
