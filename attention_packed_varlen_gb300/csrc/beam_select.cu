// Two-stage beam candidate selection on sm_103a (article "SLM 生成式高并发推理引擎：
// 延迟约束下的有效吞吐优化", section 3.3):
//
//   BF16 logits [W_in, V] -> scores read from the FP32 log-softmax over the
//   full vocabulary plus the beam's cumulative score -> the global 2W best
//   (higher score first; equal scores by lower parent, then higher logit,
//   then lower id) with their parents.
//
// The article's pruning claim -- a candidate outside the best few of its own
// group cannot reach the global 2W -- is applied to groups of logits smaller
// than a beam: tiles of 8192 consecutive logits of one row, and within a tile
// 128 interleaved groups of 64 ("sub-chunks").  A group's best score is that
// of its largest logit (the score is monotone in the logit), and 2W distinct
// groups' best scores are 2W real candidates, so the 2W-th largest group
// maximum L is at most the global 2W-th score: every global candidate lies in
// a group whose maximum scores >= L, and is itself >= L.  Only those groups
// are read again, and only their logits scoring >= L are ranked.
//
// Two kernels, the logits read once from HBM plus a few hundred small groups:
//
// 1. stream (persistent, one CTA per SM): a producer warp streams 16 KB tiles
//    into a 12-stage shared-memory ring with 1-D bulk copies (cp.async.bulk)
//    completing on mbarriers; twelve consumer warps, one per ring slot, take
//    whole tiles: the maximum of each of the tile's 128 sub-chunks (packed
//    bf16x2 max), then the tile's sum of exp(x - M_t) relative to its
//    maximum (packed f32x2 FMA and ex2).  Per tile it writes (M_t, sum) and the 128 sub-chunk maxima.
// 2. select (one CTA per SM, a programmatic dependent of the stream): every
//    CTA derives lse_b of every beam from the tile partials (a thread per
//    beam, its tiles in order) and every group's best score key into shared
//    memory, and takes as L the lower edge of the bin of 2^16 keys holding
//    the 2W-th largest key (a shared histogram); warp w of the grid then
//    re-reads, of the groups w, w + n_warps, ..., those scoring >= L -- their
//    sub-chunks scoring >= L -- and appends the logits scoring >= L to a
//    small list.  The last CTA to finish ranks that list with the full order
//    (score bins, then pairwise within a bin) and writes the 2W results.  If
//    the list would overflow (huge score ties) the last CTA ranks every logit
//    scoring >= L exactly with a radix select instead.
//
// Shapes whose group keys do not fit the select kernel's shared memory (more
// than 16,384 groups, or rows of more than 64 tiles) run a row-statistics
// kernel between the two (a warp per beam, or a CTA per beam when the groups
// are sub-chunks): lse_b, the group keys and a histogram of their upper 16
// bits in global memory; every select CTA then walks the histogram down to
// the bin holding the 2W-th largest key and takes that bin's lower edge as L.
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
constexpr int kCWarps = 12;                        // consumer warps of the stream kernel
constexpr int kVec = 4;                            // 16-byte vectors per lane and chunk
constexpr int kChunkElems = kVec * 8 * 32;         // 1024 logits per chunk
constexpr int kChunks = kTile / kChunkElems;       // 8 chunks per tile
constexpr int kStages = 12;                        // ring depth (192 KB)
constexpr int kStreamThreads = 32 * (kCWarps + 1);
constexpr int kQuarters = 4;                       // sub-chunks per lane and tile (2 chunks each)
constexpr int kSubPerTile = kQuarters * 32;        // 128 sub-chunks of 64 logits per tile
constexpr int kSelThreads = 1024;                  // select kernel threads (at most 1024: 32 warps)
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kRowThreads = 256;                   // row-statistics kernel: a warp per beam
constexpr int kRowWarps = kRowThreads / 32;
constexpr int kMaxRows = 1024;                     // W_in limit
constexpr int kUnitCap = 8192;                     // groups the exact path lists (more: it tests every group)
constexpr int kCandCap = 4096;                     // candidates the final sort holds
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kNegInf2 = 0xFF80FF80u;         // two bf16 -inf
constexpr unsigned kFull = 0xffffffffu;
static_assert(kChunks % kQuarters == 0, "a sub-chunk is a whole number of chunks");
// Consumer warp w takes the CTA's tiles w, w + kCWarps, ...; with kStages a
// multiple of kCWarps every ring slot is read by one warp only, so a warp
// waiting on a slot's "full" barrier is never two phases ahead of it (where
// the parity of the phase it wants would match an older, completed phase).
static_assert(kStages % kCWarps == 0, "each ring slot has a single consumer warp");

// misc words of the workspace
constexpr int kMiscCand = 0;     // candidates appended
constexpr int kMiscTicket = 1;   // select-kernel CTAs done
constexpr int kMiscStatus = 2;   // nonzero: a bounded wait ran out
constexpr int kMiscMaxKey = 3;   // largest group key
constexpr int kMiscWords = 4;
constexpr int kHistBins = 65536; // group keys >> 16

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

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits) { return __uint_as_float((bits & 0xFFFFu) << 16); }

__device__ __forceinline__ uint32_t f32_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_to_f32(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// A candidate as stored: bf16 bits in 32..47, token id in 0..31.
__device__ __forceinline__ unsigned long long cand_entry(uint32_t bits, uint32_t token) {
  return (static_cast<unsigned long long>(bits & 0xFFFFu) << 32) | token;
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
  bool vec_ok;             // rows 16-byte aligned: bulk copies and vector loads
  bool fused;              // the select kernel derives the row statistics itself (no row kernel, no histogram)
  // workspace
  float2* partial;         // [n_tiles] (tile maximum M_t, sum of exp(x - M_t))
  uint16_t* submax;        // [n_tiles, kSubPerTile] sub-chunk maxima (bf16 bits)
  float* lse;              // [W_in]
  uint32_t* gkeys;         // [groups] each group's best score key
  unsigned* hist;          // [kHistBins] group keys by their upper 16 bits
  ulonglong2* cand;        // [kCandCap] candidates in the global order encoding
  unsigned* misc;          // [kMiscWords]
  // outputs
  int32_t* out_token;
  int32_t* out_parent;
  float* out_score;
  int32_t* out_cand_token;
  int32_t* out_cand_parent;
  float* out_cand_score;
  float* out_lse;
};

// Tile-relative position of logit e (0..7) of run r (0..7) of sub-chunk (q, l):
// the lane l of a consumer warp reads, in chunk ch and vector v, the logits
// ch * 1024 + (v * 32 + l) * 8 + 0..7; sub-chunk (q, l) is what lane l reads in
// chunks 2q and 2q + 1.
__device__ __forceinline__ int sub_run_offset(int q, int l, int r) {
  const int ch = q * (kChunks / kQuarters) + (r >> 2), v = r & 3;
  return ch * kChunkElems + (v * 32 + l) * 8;
}

// ---------------------------------------------------------------------------
// 1. stream
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
// (ch * 1024 + (v * 32 + lane) * 8) + 0..7.  With full = false, vectors past
// the tile's n logits read as -inf.
template <bool kFullTile>
__device__ __forceinline__ void load_chunk(const uint4* slot, int ch, int lane, int n, uint4 (&r)[kVec]) {
#pragma unroll
  for (int v = 0; v < kVec; ++v) {
    const int e0 = ch * kChunkElems + (v * 32 + lane) * 8;
    r[v] = (kFullTile || e0 < n) ? slot[ch * (kChunkElems / 8) + v * 32 + lane]
                                 : make_uint4(kNegInf2, kNegInf2, kNegInf2, kNegInf2);
  }
}

__device__ __forceinline__ uint32_t hmax2_u32(uint32_t a, uint32_t b) {
  __nv_bfloat162 r = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&a), *reinterpret_cast<const __nv_bfloat162*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

// The larger of the two bf16 halves, as bf16 bits.
__device__ __forceinline__ uint32_t hmax_halves(uint32_t a) {
  return hmax2_u32(a, (a >> 16) | (a << 16)) & 0xFFFFu;
}

// One tile in a consumer warp: the 128 sub-chunk maxima (lane l holds
// sub-chunks (q, l), q = 0..3), the tile maximum, and the sum of exp(x - M).
template <bool kFullTile>
__device__ __forceinline__ void consume_tile(const uint4* slot, int n, int lane, uint32_t (&qb)[kQuarters],
                                             float& M, float& l_sum) {
  float lm = -INFINITY;
#pragma unroll
  for (int q = 0; q < kQuarters; ++q) {
    uint32_t qm = kNegInf2;
#pragma unroll
    for (int k = 0; k < kChunks / kQuarters; ++k) {
      uint4 r[kVec];
      load_chunk<kFullTile>(slot, q * (kChunks / kQuarters) + k, lane, n, r);
#pragma unroll
      for (int v = 0; v < kVec; ++v)
        qm = hmax2_u32(hmax2_u32(qm, r[v].x), hmax2_u32(hmax2_u32(r[v].y, r[v].z), r[v].w));
    }
    qb[q] = hmax_halves(qm);
    lm = fmaxf(lm, bf16_bits_to_f32(qb[q]));
  }
  M = warp_max(lm);
  float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
  if (M > -INFINITY) {
    const float cc = -M * kLog2e;
#pragma unroll 2
    for (int ch = 0; ch < kChunks; ++ch) {
      uint4 r[kVec];
      load_chunk<kFullTile>(slot, ch, lane, n, r);
      chunk_exp_sum(r, cc, s0, s1, s2, s3);
    }
  }
  l_sum = (s0 + s1) + (s2 + s3);
}

// Consumer warp cw takes the CTA's tiles cw, cw + kCWarps, ... whole, so the
// warps work on different tiles and no warp waits for another; each ring slot
// belongs to one warp.
__device__ void stream_consumer(const Params& p, StreamSmem& sh, int cw, int lane) {
  const int step = kCWarps * gridDim.x;
  for (int i = cw, t = blockIdx.x + cw * gridDim.x; t < p.n_tiles; i += kCWarps, t += step) {
    const int s = i % kStages;
    const int b = t / p.n_tpr, c = t - b * p.n_tpr;
    const int n = min(kTile, p.V - c * kTile);
    const bool ok = mbar_wait(&sh.full[s], (i / kStages) & 1, &sh.abort);
    if (!__all_sync(kFull, ok)) break;
    const uint4* slot = &sh.ring[s][0];
    uint32_t qb[kQuarters];
    float M, l;
    if (n == kTile) consume_tile<true>(slot, n, lane, qb, M, l);
    else consume_tile<false>(slot, n, lane, qb, M, l);
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.empty[s]);  // the slot's data is no longer read
    l = warp_sum(l);
    if (lane == 0) p.partial[t] = make_float2(M, l);
    uint16_t* sm = p.submax + static_cast<int64_t>(t) * kSubPerTile;
#pragma unroll
    for (int q = 0; q < kQuarters; ++q) sm[q * 32 + lane] = static_cast<uint16_t>(qb[q]);
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
  // Global memory (the logits, and the workspace an earlier call's select
  // kernel reads) only after everything before this kernel is done; as an
  // ordinary launch it starts after that anyway, and the wait returns at once.
  grid_dep_wait();
  if (threadIdx.x == 0 && blockIdx.x == 0)
    for (int i = 0; i < kMiscWords; ++i) p.misc[i] = 0u;  // read by the select kernel after this grid ends
  if (!p.fused) {  // this CTA's slice of the group-key histogram (filled by the row kernel after this grid ends)
    const int per = (kHistBins + gridDim.x - 1) / gridDim.x;
    const int end = min(kHistBins, (static_cast<int>(blockIdx.x) + 1) * per);
    for (int i = blockIdx.x * per + threadIdx.x; i < end; i += kStreamThreads) p.hist[i] = 0u;
  }
  __syncthreads();
  grid_dep_launch();
  if (warp == 0) stream_producer(p, sh, lane);
  else stream_consumer(p, sh, warp - 1, lane);
  __syncthreads();
  if (threadIdx.x == 0 && sh.abort) atomicOr(p.misc + kMiscStatus, 1u);
}

// ---------------------------------------------------------------------------
// Block primitives of the select kernel (kSelThreads threads)
// ---------------------------------------------------------------------------
struct Scratch {
  unsigned hist[256];
  unsigned long long wu64[2][kSelWarps];
  int wint[kSelWarps];
  uint32_t wkey[kSelWarps];
  int digit, above, in_bin, counter, flag, dstar;
  unsigned long long u64;
};

// Block-wide exclusive prefix sum and total.  After one barrier every warp
// reads the warps' totals, one word per lane, and scans them with shuffles:
// two barriers, and no thread loops over the 32 totals (which costs ~1,000
// cycles of the shared-memory pipe per call with 1024 threads).
__device__ __forceinline__ int block_scan_excl(int v, int* total, Scratch& sh) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int x = warp_inclusive_scan(v, lane);
  __syncthreads();  // earlier readers of sh.wint are done
  if (lane == 31) sh.wint[w] = x;
  __syncthreads();
  const int y = (lane < kSelWarps) ? sh.wint[lane] : 0;
  const int inc = warp_inclusive_scan(y, lane);
  *total = __shfl_sync(kFull, inc, 31);
  return __shfl_sync(kFull, inc - y, w) + x - v;
}

// Block-wide maximum (two barriers, as above).
__device__ __forceinline__ uint32_t block_max_u32(uint32_t v, Scratch& sh) {
  const int lane = threadIdx.x & 31;
  v = warp_max_u32(v);
  __syncthreads();
  if (lane == 0) sh.wkey[threadIdx.x >> 5] = v;
  __syncthreads();
  return warp_max_u32((lane < kSelWarps) ? sh.wkey[lane] : 0u);
}

// k-th largest (1-based, counting repeats) of the 64-bit keys all threads
// visit with for_each(f).  Each pass histograms the keys in the live range
// [lo, hi] by the 8 bits below the range's leading bit and narrows the range
// to the bin holding the k-th key; a bin with a single key ends it.
template <class ForEach>
__device__ unsigned long long block_kth(ForEach for_each, int k, Scratch& sh, unsigned (*whist)[256]) {
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
  if (w == 0) {
    const unsigned long long l = warp_min_u64((lane < kSelWarps) ? sh.wu64[0][lane] : ~0ull),
                             h = warp_max_u64((lane < kSelWarps) ? sh.wu64[1][lane] : 0ull);
    if (lane == 0) {
      sh.wu64[0][0] = l;
      sh.wu64[1][0] = h;
    }
  }
  __syncthreads();
  lo = sh.wu64[0][0];
  hi = sh.wu64[1][0];
  while (lo < hi) {
    const int sft = max(0, 64 - __clzll(hi - lo) - 8);
    for (int i = threadIdx.x; i < kSelWarps * 256; i += kSelThreads) (&whist[0][0])[i] = 0u;
    __syncthreads();
    const unsigned long long lo_c = lo, hi_c = hi;
    for_each([&](unsigned long long key) {
      if (key >= lo_c && key <= hi_c) atomicAdd(&whist[w][static_cast<uint32_t>((key - lo_c) >> sft)], 1u);
    });
    __syncthreads();
    if (threadIdx.x < 256) {
      unsigned s = 0;
      for (int i = 0; i < kSelWarps; ++i) s += whist[i][threadIdx.x];
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

// Descending bitonic sort of ent[0, n_pow2) (the rare exact path only).
__device__ void block_sort_desc(ulonglong2* ent, int n_pow2) {
  for (int size = 2; size <= n_pow2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      __syncthreads();
      for (int t = threadIdx.x; t < n_pow2 / 2; t += kSelThreads) {
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
// Row statistics for shapes beyond the fused path (a warp per beam)
// ---------------------------------------------------------------------------
// Score key fl32(cum + fl32(x - lse)), order-preserving.
__device__ __forceinline__ uint32_t score_key_x(float x, float cum, float lse) {
  return f32_key(__fadd_rn(cum, __fsub_rn(x, lse)));
}

// lse_b from the beam's tiles (fixed order: lane j holds tile j, then the
// warp's butterfly reductions), then the key of every group of the beam --
// its tiles when there are at least K tiles in all, else its sub-chunks --
// into gkeys, the histogram of the keys' upper 16 bits, and the largest key.
// One red.add per distinct histogram bin among the warp's lanes.
__device__ __forceinline__ void hist_add(unsigned* hist, uint32_t key, bool valid) {
  const uint32_t bin = valid ? (key >> 16) : 0xFFFFFFFFu;
  const unsigned peers = __match_any_sync(kFull, bin);
  if (valid && (threadIdx.x & 31) == static_cast<unsigned>(__ffs(peers) - 1)) red_add(hist + bin, __popc(peers));
}

__global__ void __launch_bounds__(kRowThreads) rowstat_kernel(const Params p) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bool sub_level = p.n_tiles < p.K;
  // tile groups: a warp per beam; sub-chunk groups: a CTA per beam
  const int b = sub_level ? static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x) * kRowWarps + warp;
  grid_dep_wait();
  grid_dep_launch();
  if (b >= p.W_in) return;
  const int nt = p.n_tpr;
  const float2* P = p.partial + static_cast<int64_t>(b) * nt;
  const float cum = __ldg(p.cum + b);
  float M = -INFINITY;
  for (int j = lane; j < nt; j += 32) {
    const float2 q = __ldcg(P + j);
    if (q.y > 0.f) M = fmaxf(M, q.x);
  }
  M = warp_max(M);
  float L = 0.f;
  for (int j = lane; j < nt; j += 32) {
    const float2 q = __ldcg(P + j);
    if (q.y > 0.f) L += q.y * ex2((q.x - M) * kLog2e);
  }
  L = warp_sum(L);
  const float lse = (L > 0.f) ? M + logf(L) : -INFINITY;
  if (lane == 0 && (!sub_level || warp == 0)) {
    p.lse[b] = lse;
    if (p.out_lse) p.out_lse[b] = lse;
  }
  uint32_t kmax = 0u;
  if (!sub_level) {
    for (int j0 = 0; j0 < nt; j0 += 32) {
      const int j = j0 + lane;
      const bool valid = j < nt;
      const uint32_t key = valid ? score_key_x(__ldcg(&P[j].x), cum, lse) : 0u;
      if (valid) p.gkeys[static_cast<int64_t>(b) * nt + j] = key;
      hist_add(p.hist, key, valid);
      kmax = max(kmax, key);
    }
  } else {
    const int n = nt * kSubPerTile;
    const uint16_t* sm = p.submax + static_cast<int64_t>(b) * n;
    uint32_t* gk = p.gkeys + static_cast<int64_t>(b) * n;
    for (int i0 = warp * 32; i0 < n; i0 += kRowThreads) {
      const int i = i0 + lane;
      const bool valid = i < n;
      const uint32_t key = valid ? score_key_x(bf16_bits_to_f32(__ldcg(sm + i)), cum, lse) : 0u;
      if (valid) gk[i] = key;
      hist_add(p.hist, key, valid);
      kmax = max(kmax, key);
    }
  }
  kmax = warp_max_u32(kmax);
  if (lane == 0) atomicMax(p.misc + kMiscMaxKey, kmax);
}

// ---------------------------------------------------------------------------
// 2. select
// ---------------------------------------------------------------------------
constexpr int kBins = 4096;                      // final ranking bins
constexpr int kKeyCap = 16384;                   // fused path: group keys held in shared memory
constexpr int kFusedMaxTpr = 64;                 // fused path: tiles per row (a thread per beam sums them)
constexpr int kUnitWords = 16384;                // ballot words: groups up to 524,288
constexpr int kBinsPerThread = kBins / kSelThreads;
constexpr int kCandPer = kCandCap / kSelThreads;  // candidates per thread in the final ranking
static_assert(kBins % kSelThreads == 0, "whole bins per thread");

// Dynamic shared memory of the select kernel.
struct SelSmem {
  float lse[kMaxRows];
  float cum[kMaxRows];
  uint32_t keys[kKeyCap];     // fused path: every group's best score key
  int units[kUnitCap];        // the exact path: groups scoring >= L (tiles, or sub-chunks t * 128 + s)
  unsigned bins[kBins];
  int fill[kBins];
  int rtok[2048], rpar[2048];  // the K results, written out together
  float rsc[2048];
  union {
    ulonglong2 ent[kCandCap];   // the last CTA's candidates grouped by score bin; the exact path's result
    unsigned whist[kSelWarps][256];  // the exact path's radix histograms
    uint32_t words[kUnitWords];      // ballot words of the groups scoring >= L
  } u;
  Scratch sc;
};
static_assert(sizeof(SelSmem) <= 232448, "the select kernel's shared memory fits one CTA");

// Result r of the global order into shared memory; error = true: -1 ids and NaN scores.
__device__ __forceinline__ void stage_result(SelSmem& sm, int r, const ulonglong2& g, bool error = false) {
  sm.rtok[r] = error ? -1 : static_cast<int>(0xFFFFFFFFull - g.y);
  sm.rpar[r] = error ? -1 : 0xFFFF - static_cast<int>((g.x >> 16) & 0xFFFFull);
  sm.rsc[r] = error ? __int_as_float(0x7fc00000) : key_to_f32(static_cast<uint32_t>(g.x >> 32));
}

__device__ __forceinline__ void write_results(const Params& p, const SelSmem& sm) {
  __syncthreads();
  for (int r = threadIdx.x; r < p.K; r += kSelThreads) {
    if (r < p.W) {
      p.out_token[r] = sm.rtok[r];
      p.out_parent[r] = sm.rpar[r];
      p.out_score[r] = sm.rsc[r];
    }
    if (p.out_cand_token) p.out_cand_token[r] = sm.rtok[r];
    if (p.out_cand_parent) p.out_cand_parent[r] = sm.rpar[r];
    if (p.out_cand_score) p.out_cand_score[r] = sm.rsc[r];
  }
}

__device__ __forceinline__ void write_errors(const Params& p, SelSmem& sm) {
  for (int r = threadIdx.x; r < p.K; r += kSelThreads) stage_result(sm, r, make_ulonglong2(0ull, 0ull), true);
  write_results(p, sm);
}

// Eight logits of row b at columns col .. col + 7 (as four bf16x2 words);
// columns at or past V read as -inf.
__device__ __forceinline__ uint4 load_run(const Params& p, int b, int col) {
  const uint16_t* row = p.logits + static_cast<int64_t>(b) * p.V;
  if (p.vec_ok && col + 8 <= p.V) return __ldcs(reinterpret_cast<const uint4*>(row + col));
  uint32_t w[4];
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    const uint32_t lo = (col + 2 * h < p.V) ? row[col + 2 * h] : 0xFF80u;
    const uint32_t hi = (col + 2 * h + 1 < p.V) ? row[col + 2 * h + 1] : 0xFF80u;
    w[h] = lo | (hi << 16);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Fused path: every select CTA derives the row statistics itself from the
// stream kernel's tile partials.  One coalesced pass loads every tile's
// (M_t, sum) -- and, for sub-chunk groups, every sub-chunk maximum -- into
// shared memory; a thread per beam then takes the beam's tiles in order for
// lse_b (maximum, then the sum of the rescaled sums) and the group keys are
// scored in place: the beam's tile maxima by that thread (tile groups), or
// every sub-chunk maximum once all lse are known (sub-chunk groups).  The
// arithmetic is the same in every CTA, so all CTAs hold the same lse and keys.
__device__ uint32_t fused_row_stats(const Params& p, SelSmem& sm, bool tile_level, int n_groups) {
  const int nt = p.n_tpr;
  uint32_t mk = 0u;  // the largest key
  // tile groups: M_t in the keys array (scored in place), sums in the union;
  // sub-chunk groups (fewer than 2W <= 2048 tiles): both in the union
  uint32_t* Mt = tile_level ? sm.keys : sm.u.words;
  uint32_t* St = tile_level ? sm.u.words : sm.u.words + kUnitWords / 2;
  for (int t = threadIdx.x; t < p.n_tiles; t += kSelThreads) {
    const float2 q = __ldcg(p.partial + t);
    Mt[t] = __float_as_uint(q.x);
    St[t] = __float_as_uint(q.y);
  }
  if (!tile_level)
    for (int g = threadIdx.x; g < n_groups; g += kSelThreads) sm.keys[g] = __ldcg(p.submax + g);
  __syncthreads();
  for (int b = threadIdx.x; b < p.W_in; b += kSelThreads) {
    const uint32_t* m = Mt + b * nt;
    const uint32_t* sb = St + b * nt;
    float M = -INFINITY;
#pragma unroll 4
    for (int j = 0; j < nt; ++j)
      if (__uint_as_float(sb[j]) > 0.f) M = fmaxf(M, __uint_as_float(m[j]));
    float L = 0.f;
#pragma unroll 4
    for (int j = 0; j < nt; ++j) {
      const float sj = __uint_as_float(sb[j]);
      if (sj > 0.f) L += sj * ex2((__uint_as_float(m[j]) - M) * kLog2e);
    }
    const float lse = (L > 0.f) ? M + logf(L) : -INFINITY;
    sm.lse[b] = lse;
    if (blockIdx.x == 0 && p.out_lse) p.out_lse[b] = lse;
    if (tile_level) {
      const float cum = sm.cum[b];
      for (int j = 0; j < nt; ++j) {
        const uint32_t key = score_key_x(__uint_as_float(m[j]), cum, lse);
        sm.keys[b * nt + j] = key;
        mk = max(mk, key);
      }
    }
  }
  if (!tile_level) {
    __syncthreads();
    for (int g = threadIdx.x; g < n_groups; g += kSelThreads) {
      const int b = (g / kSubPerTile) / nt;
      const uint32_t key = score_key_x(bf16_bits_to_f32(sm.keys[g]), sm.cum[b], sm.lse[b]);
      sm.keys[g] = key;
      mk = max(mk, key);
    }
  }
  return block_max_u32(mk, sm.sc);  // its barriers also publish the keys
}

// Fused path: the lower edge of the bin of 2^16 keys that holds the K-th
// largest group key, from a histogram of the keys' upper 16 bits counted down
// from the largest key's (kBins bins in shared memory), or false when the
// K-th key lies further down than kBins bins (then the caller selects
// exactly).  `hist` is zero on entry.
__device__ bool fused_threshold(const SelSmem& sm, int* hist, int n_groups, int K, uint32_t maxkey, Scratch& sh,
                                uint32_t* Lk) {
  const int tid = threadIdx.x;
  const uint32_t top = maxkey >> 16;
  if (tid == 0) sh.dstar = -1;
  for (int g = tid; g < n_groups; g += kSelThreads) {
    const uint32_t d = top - (sm.keys[g] >> 16);
    if (d < static_cast<uint32_t>(kBins)) atomicAdd(hist + d, 1);
  }
  __syncthreads();
  const int d0 = tid * kBinsPerThread;
  int c[kBinsPerThread], local = 0;
#pragma unroll
  for (int i = 0; i < kBinsPerThread; ++i) {
    c[i] = hist[d0 + i];
    local += c[i];
  }
  int total;
  int ex = block_scan_excl(local, &total, sh);
  if (ex < K && ex + local >= K) {
#pragma unroll
    for (int i = 0; i < kBinsPerThread; ++i) {
      if (ex < K && ex + c[i] >= K) sh.dstar = d0 + i;
      ex += c[i];
    }
  }
  __syncthreads();
  const int dstar = sh.dstar;
  if (dstar < 0) return false;
  *Lk = (top - static_cast<uint32_t>(dstar)) << 16;
  return true;
}

template <bool kFused>
__global__ void __launch_bounds__(kSelThreads, 1) select_kernel(const Params p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  SelSmem& sm = *reinterpret_cast<SelSmem*>(smem_raw);
  Scratch& sh = sm.sc;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = p.K, nt = p.n_tpr;
  for (int i = tid; i < kBins; i += kSelThreads) {
    sm.bins[i] = 0u;
    sm.fill[i] = 0;
  }
  // Global memory only after the wait: the stream kernel's products, and the
  // cumulative scores, which an earlier kernel still running may be writing.
  grid_dep_wait();
  for (int b = tid; b < p.W_in; b += kSelThreads) sm.cum[b] = __ldcg(p.cum + b);
  // the groups: tiles when there are at least K of them, else sub-chunks
  const bool tile_level = p.n_tiles >= K;
  const int n_groups = tile_level ? p.n_tiles : p.n_tiles * kSubPerTile;
  uint32_t maxkey;
  if constexpr (kFused) {
    maxkey = fused_row_stats(p, sm, tile_level, n_groups);
  } else {
    for (int b = tid; b < p.W_in; b += kSelThreads) sm.lse[b] = __ldcg(p.lse + b);
    maxkey = __ldcg(p.misc + kMiscMaxKey);
  }

  // L: the lower edge of the bin of 2^16 keys that holds the K-th largest
  // group key -- at most that key, so at least K groups score >= L.  Fused
  // path: from a histogram of the keys in shared memory (or exactly that key,
  // by radix select, when it lies far below the largest); otherwise: the
  // global histogram walked down from the largest key's bin.  At most K
  // groups: all of them.
  uint32_t Lk = 0u;
  if (kFused && n_groups > K) {
    if (!fused_threshold(sm, sm.fill, n_groups, K, maxkey, sh, &Lk))
      Lk = static_cast<uint32_t>(block_kth(
          [&](auto f) {
            for (int g = tid; g < n_groups; g += kSelThreads) f(static_cast<unsigned long long>(sm.keys[g]));
          },
          K, sh, sm.u.whist));
  } else if (n_groups > K) {
    int carry = 0;
    if (tid == 0) sh.dstar = -1;
    for (int top = static_cast<int>(maxkey >> 16); top >= 0; top -= kSelThreads) {
      const int bin = top - tid;
      const int c = (bin >= 0) ? static_cast<int>(__ldcg(p.hist + bin)) : 0;
      int total;
      const int ex = block_scan_excl(c, &total, sh);
      if (carry + ex < K && carry + ex + c >= K) sh.dstar = bin;
      carry += total;
      if (carry >= K) break;  // uniform
    }
    __syncthreads();
    if (sh.dstar >= 0) Lk = static_cast<uint32_t>(sh.dstar) << 16;
  }

  // Read back the groups scoring >= L and append their logits scoring >= L.
  // Warp gw of the grid takes groups gw, gw + n_gw, gw + 2 n_gw, ...: each
  // lane tests one group's key per step and the warp re-reads the groups that
  // pass one by one, so the ~2W groups spread over the grid's warps without a
  // shared list.  Per group, a warp handles up to four of its sub-chunks
  // scoring >= L at once, eight lanes each, one 16-byte run of eight logits
  // per lane.
  auto group_key = [&](int g) -> uint32_t { return kFused ? sm.keys[g] : __ldcg(p.gkeys + g); };
  {
    const int gw = blockIdx.x * kSelWarps + warp, n_gw = gridDim.x * kSelWarps;
    for (int g0 = gw; g0 < n_groups; g0 += 32 * n_gw) {
      const int gl = g0 + lane * n_gw;
      unsigned pending = __ballot_sync(kFull, gl < n_groups && group_key(gl) >= Lk);
      while (pending) {
        const int g = g0 + (__ffs(pending) - 1) * n_gw;
        pending &= pending - 1u;
        const int t = tile_level ? g : g / kSubPerTile;
        const int b = t / nt, c = t - b * nt;
        const float cum = sm.cum[b], lse = sm.lse[b];
        // the tile's sub-chunks scoring >= L, as four lane masks (q = 0..3)
        unsigned mq[kQuarters];
        if (tile_level) {
          const uint16_t* smx = p.submax + static_cast<int64_t>(t) * kSubPerTile;
#pragma unroll
          for (int q = 0; q < kQuarters; ++q)
            mq[q] = __ballot_sync(kFull, score_key_x(bf16_bits_to_f32(__ldcg(smx + q * 32 + lane)), cum, lse) >= Lk);
        } else {
          const int s = g - t * kSubPerTile;
#pragma unroll
          for (int q = 0; q < kQuarters; ++q) mq[q] = (q == s / 32) ? (1u << (s % 32)) : 0u;
        }
        const int n0 = __popc(mq[0]), n1 = __popc(mq[1]), n2 = __popc(mq[2]);
        const int n_sub = n0 + n1 + n2 + __popc(mq[3]);
        for (int base = 0; base < n_sub; base += 4) {
          const int j = base + (lane >> 3), r = lane & 7;  // sub-chunk j of the list, run r
          int cnt = 0;
          uint4 x = make_uint4(kNegInf2, kNegInf2, kNegInf2, kNegInf2);
          int col = 0;
          if (j < n_sub) {
            int q = 0, k = j;
            unsigned m = mq[0];
            if (k >= n0) { k -= n0; q = 1; m = mq[1];
              if (k >= n1) { k -= n1; q = 2; m = mq[2];
                if (k >= n2) { k -= n2; q = 3; m = mq[3]; } } }
            for (int i = 0; i < k; ++i) m &= m - 1u;  // drop the k lowest set bits
            const int l = __ffs(m) - 1;
            col = c * kTile + sub_run_offset(q, l, r);
            x = load_run(p, b, col);
          }
          const uint32_t wd[4] = {x.x, x.y, x.z, x.w};
          uint32_t keys[8];
#pragma unroll
          for (int h = 0; h < 8; ++h) {
            keys[h] = score_key_x(bf16_bits_to_f32((h & 1) ? (wd[h >> 1] >> 16) : (wd[h >> 1] & 0xFFFFu)), cum, lse);
            cnt += (j < n_sub && keys[h] >= Lk);
          }
          const int incl = warp_inclusive_scan(cnt, lane);
          const int total = __shfl_sync(kFull, incl, 31);
          if (total == 0) continue;
          unsigned pos0 = 0;
          if (lane == 0) pos0 = atomicAdd(p.misc + kMiscCand, static_cast<unsigned>(total));
          int pos = static_cast<int>(__shfl_sync(kFull, pos0, 0)) + incl - cnt;
#pragma unroll
          for (int h = 0; h < 8; ++h) {
            if (j < n_sub && keys[h] >= Lk) {
              if (pos < kCandCap) {
                const uint32_t bits = (h & 1) ? (wd[h >> 1] >> 16) : (wd[h >> 1] & 0xFFFFu);
                p.cand[pos] = global_entry(keys[h], static_cast<uint32_t>(b),
                                           cand_entry(bits, static_cast<uint32_t>(col + h)));
              }
              ++pos;
            }
          }
        }
      }
    }
  }

  // the last CTA to finish ranks the list
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    sh.flag = (atom_add_acq_rel(p.misc + kMiscTicket, 1u) == gridDim.x - 1);
  }
  __syncthreads();
  grid_dep_launch();  // the next kernel may start its setup while the last CTA ranks
  if (!sh.flag) return;

  if (__ldcg(p.misc + kMiscStatus) != 0u) {
    write_errors(p, sm);
    return;
  }
  const int n_cand = static_cast<int>(__ldcg(p.misc + kMiscCand));
  if (n_cand <= kCandCap) {
    if (n_cand < K) {  // cannot happen: every group scoring >= L holds one candidate
      write_errors(p, sm);
      return;
    }
    // Rank by bin: an entry's place is the count of the entries in the bins
    // above its own (bins of the score key counted down from the largest,
    // all scores >= L spread over kBins bins) plus its rank among the
    // entries of its own bin.
    const unsigned long long range = static_cast<unsigned long long>(maxkey - min(Lk, maxkey));
    const int s2 = max(0, 64 - __clzll(range + 1ull) - 12);  // (range >> s2) < kBins
    auto bin_of = [&](unsigned long long hi) -> uint32_t {
      const uint32_t skey = static_cast<uint32_t>(hi >> 32);
      return min(static_cast<uint32_t>(static_cast<unsigned long long>(maxkey - min(skey, maxkey)) >> s2),
                 static_cast<uint32_t>(kBins - 1));
    };
    // the candidates, up to kCandPer per thread, held in registers
    unsigned long long ch[kCandPer], cl[kCandPer];
#pragma unroll
    for (int k = 0; k < kCandPer; ++k) {
      const int i = tid + k * kSelThreads;
      ch[k] = (i < n_cand) ? __ldcg(&p.cand[i].x) : 0ull;
      cl[k] = (i < n_cand) ? __ldcg(&p.cand[i].y) : 0ull;
    }
#pragma unroll
    for (int k = 0; k < kCandPer; ++k)
      if (tid + k * kSelThreads < n_cand) atomicAdd(&sm.bins[bin_of(ch[k])], 1u);
    __syncthreads();
    // bins -> first position of each bin (fill[] keeps the counts)
    {
      const int d0 = tid * kBinsPerThread;
      int cnt = 0;
#pragma unroll
      for (int i = 0; i < kBinsPerThread; ++i) cnt += static_cast<int>(sm.bins[d0 + i]);
      int total;
      int c = block_scan_excl(cnt, &total, sh);
#pragma unroll
      for (int i = 0; i < kBinsPerThread; ++i) {
        const int v = static_cast<int>(sm.bins[d0 + i]);
        sm.fill[d0 + i] = v;
        sm.bins[d0 + i] = static_cast<unsigned>(c);
        c += v;
      }
    }
    __syncthreads();
    // the entries themselves, grouped by bin (bins in score order)
#pragma unroll
    for (int k = 0; k < kCandPer; ++k)
      if (tid + k * kSelThreads < n_cand)
        sm.u.ent[atomicAdd(&sm.bins[bin_of(ch[k])], 1u)] = make_ulonglong2(ch[k], cl[k]);  // bins[d]: one past the bin
    __syncthreads();
    // Each entry's rank: the entries of the bins above, plus those of its own
    // bin that come before it.  A warp's entries are neighbours in the grouped
    // list, mostly of one bin, so its lanes read the same entries together.
    for (int pos = tid; pos < n_cand; pos += kSelThreads) {
      const ulonglong2 e = sm.u.ent[pos];
      const uint32_t d = bin_of(e.x);
      const int g1 = static_cast<int>(sm.bins[d]), g0 = g1 - sm.fill[d];
      int rank = g0;
      for (int j = g0; j < g1; ++j) rank += entry_greater(sm.u.ent[j], e);
      if (rank < K) stage_result(sm, rank, e);
    }
    write_results(p, sm);
    return;
  }

  // Huge score ties: every logit scoring >= L, ranked exactly.  The groups
  // scoring >= L are listed in group order (each warp reads a contiguous
  // range once, keeping one ballot word per 32 groups in shared memory) or,
  // when they overflow the list, every group is tested; all of their logits
  // are visited.
  int n_found;
  {
    uint32_t* words = sm.u.words;
    const int n_words = min((n_groups + 31) >> 5, kUnitWords);  // more groups: the exact path
    const int per = (n_words + kSelWarps - 1) / kSelWarps;  // words per warp
    const int w_lo = min(n_words, warp * per), w_hi = min(n_words, w_lo + per);
    int cnt = 0;
    for (int w0 = w_lo; w0 < w_hi; w0 += 8) {
      uint32_t k8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int g = (w0 + i) * 32 + lane;
        k8[i] = (w0 + i < w_hi && g < n_groups) ? group_key(g) : 0u;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int g = (w0 + i) * 32 + lane;
        const unsigned bal = __ballot_sync(kFull, w0 + i < w_hi && g < n_groups && k8[i] >= Lk);
        if (w0 + i < w_hi && lane == 0) words[w0 + i] = bal;
        cnt += __popc(bal);
      }
    }
    // the warps' counts in warp order: lane 0 of each warp contributes its count
    int pos = block_scan_excl(lane == 0 ? cnt : 0, &n_found, sh);
    pos = __shfl_sync(kFull, pos, 0);
    for (int wd = w_lo; wd < w_hi; ++wd) {
      const unsigned bal = words[wd];
      const int at = pos + __popc(bal & ((1u << lane) - 1u));
      if (((bal >> lane) & 1u) && at < kUnitCap) sm.units[at] = wd * 32 + lane;
      pos += __popc(bal);
    }
    __syncthreads();
  }
  const int n_units = min(n_found, kUnitCap);
  const bool unit_over = n_found > kUnitCap || ((n_groups + 31) >> 5) > kUnitWords;

  const int group_size = tile_level ? kTile : 64;
  const int n_scan = unit_over ? n_groups : n_units;
  auto for_each_entry = [&](auto f) {
    for (int u = 0; u < n_scan; ++u) {
      const int g = unit_over ? u : sm.units[u];
      if (unit_over && group_key(g) < Lk) continue;  // uniform: every thread tests the same key
      const int t = tile_level ? g : g / kSubPerTile;
      const int b = t / nt, c = t - b * nt;
      const float cum = sm.cum[b], lse = sm.lse[b];
      const uint16_t* row = p.logits + static_cast<int64_t>(b) * p.V;
      for (int e = tid; e < group_size; e += kSelThreads) {
        int off;
        if (tile_level) {
          off = e;
        } else {
          const int s = g - t * kSubPerTile;
          off = sub_run_offset(s / 32, s % 32, e >> 3) + (e & 7);
        }
        const int col = c * kTile + off;
        if (col >= p.V) continue;
        const uint32_t bits = __ldcg(row + col);
        const uint32_t key = score_key_x(bf16_bits_to_f32(bits), cum, lse);
        if (key >= Lk) f(global_entry(key, static_cast<uint32_t>(b), cand_entry(bits, static_cast<uint32_t>(col))));
      }
    }
  };
  const unsigned long long kth_hi =
      block_kth([&](auto f) { for_each_entry([&](const ulonglong2& g) { f(g.x); }); }, K, sh, sm.u.whist);
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
      K - above, sh, sm.u.whist);
  if (tid == 0) sh.counter = 0;
  __syncthreads();
  for_each_entry([&](const ulonglong2& g) {
    if (g.x > kth_hi || (g.x == kth_hi && g.y >= kth_lo)) {
      const int pos = atomicAdd(&sh.counter, 1);
      if (pos < kCandCap) sm.u.ent[pos] = g;
    }
  });
  __syncthreads();
  const int n2 = next_pow2(max(K, 2));
  for (int i = K + tid; i < n2; i += kSelThreads) sm.u.ent[i] = make_ulonglong2(0ull, 0ull);
  block_sort_desc(sm.u.ent, n2);
  for (int r = tid; r < K; r += kSelThreads) stage_result(sm, r, sm.u.ent[r]);
  write_results(p, sm);
}

}  // namespace sel

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
namespace {

struct SelLayout {
  int n_tpr;
  size_t off_partial, off_submax, off_lse, off_gkeys, off_hist, off_cand, off_misc, total;
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

bool sel_layout(int W_in, int V, int W, SelLayout* L) {
  if (W_in <= 0 || V <= 0 || W <= 0) return false;
  const int64_t K = 2 * static_cast<int64_t>(W);
  if (K > 2048 || K > V || W_in > sel::kMaxRows || V >= (1 << 24)) return false;
  L->n_tpr = (V + sel::kTile - 1) / sel::kTile;
  const size_t n_tiles = size_t(W_in) * L->n_tpr;
  size_t o = 0;
  L->off_partial = o; o = align256(o + sizeof(float2) * n_tiles);
  L->off_submax = o;  o = align256(o + sizeof(uint16_t) * n_tiles * sel::kSubPerTile);
  L->off_lse = o;     o = align256(o + sizeof(float) * size_t(W_in));
  L->off_gkeys = o;   o = align256(o + sizeof(uint32_t) * n_tiles * sel::kSubPerTile);
  L->off_hist = o;    o = align256(o + sizeof(unsigned) * size_t(sel::kHistBins));
  L->off_cand = o;    o = align256(o + sizeof(ulonglong2) * size_t(sel::kCandCap));
  L->off_misc = o;    o = align256(o + sizeof(unsigned) * sel::kMiscWords);
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
  p.vec_ok = (V % 8 == 0) && ((reinterpret_cast<uintptr_t>(logits) & 15) == 0);
  {
    const int64_t n_groups = p.n_tiles >= p.K ? int64_t(p.n_tiles) : int64_t(p.n_tiles) * sel::kSubPerTile;
    p.fused = L.n_tpr <= sel::kFusedMaxTpr && n_groups <= sel::kKeyCap;
  }
  p.partial = reinterpret_cast<float2*>(ws + L.off_partial);
  p.submax = reinterpret_cast<uint16_t*>(ws + L.off_submax);
  p.lse = reinterpret_cast<float*>(ws + L.off_lse);
  p.gkeys = reinterpret_cast<uint32_t*>(ws + L.off_gkeys);
  p.hist = reinterpret_cast<unsigned*>(ws + L.off_hist);
  p.cand = reinterpret_cast<ulonglong2*>(ws + L.off_cand);
  p.misc = reinterpret_cast<unsigned*>(ws + L.off_misc);
  p.out_token = out_token;
  p.out_parent = out_parent;
  p.out_score = out_score;
  p.out_cand_token = out_cand_token;
  p.out_cand_parent = out_cand_parent;
  p.out_cand_score = out_cand_score;
  p.out_lse = out_lse;

  // The stream kernel is an ordinary launch: it starts once everything before
  // it on the stream is done, a previous call still reading this workspace
  // included (launched as a programmatic dependent of a decode attention, its
  // 152 early CTAs held the SMs the attention leaves free and the W = 400
  // decode loop ran 6 us slower).  The kernels after it are programmatic
  // dependents: each sets itself up early and waits (griddepcontrol.wait)
  // before it touches global memory.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const size_t smem_stream = sizeof(sel::StreamSmem);
  cudaError_t e = cudaFuncSetAttribute(sel::stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem_stream));
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3(std::min(sm_count(), p.n_tiles));
  cfg.blockDim = dim3(sel::kStreamThreads);
  cfg.dynamicSmemBytes = smem_stream;
  cfg.numAttrs = 0;
  e = cudaLaunchKernelEx(&cfg, sel::stream_kernel, p);
  if (e != cudaSuccess) return e;
  cfg.numAttrs = 1;

  if (!p.fused) {
    cfg.gridDim = dim3(p.n_tiles < p.K ? W_in : (W_in + sel::kRowWarps - 1) / sel::kRowWarps);
    cfg.blockDim = dim3(sel::kRowThreads);
    cfg.dynamicSmemBytes = 0;
    e = cudaLaunchKernelEx(&cfg, sel::rowstat_kernel, p);
    if (e != cudaSuccess) return e;
  }

  const size_t smem_sel = sizeof(sel::SelSmem);
  auto* select = p.fused ? sel::select_kernel<true> : sel::select_kernel<false>;
  e = cudaFuncSetAttribute(select, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_sel));
  if (e != cudaSuccess) return e;
  // One CTA per SM.  (With the row kernel a narrow selection ran faster on 32
  // CTAs; with the row statistics in the select kernel, more CTAs finish the
  // re-read sooner: 18.3 against 19.3 us at W = 100, 13.4 against 15.0 us on
  // its first step.)
  cfg.gridDim = dim3(sm_count());
  cfg.blockDim = dim3(sel::kSelThreads);
  cfg.dynamicSmemBytes = smem_sel;
  return cudaLaunchKernelEx(&cfg, select, p);
}

}  // namespace slm
