// C ABI of the attention hot path (declared in include/slm_attn.h): argument
// validation, TMA tensor-map encoding, schedule and kernel launches.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include <cuda.h>
#include <cuda_runtime.h>

#include "attn_fwd.cuh"
#include "slm_attn.h"
#include "slm_internal.h"

// Builds with -DSLM_NVTX mark every entry point as an NVTX range (host side)
// for timeline tools; other builds have no NVTX dependency at all.
#ifdef SLM_NVTX
#include <nvtx3/nvToolsExt.h>
namespace {
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};
}  // namespace
#define SLM_RANGE(name) NvtxRange slm_nvtx_range_(name)
#else
#define SLM_RANGE(name) ((void)0)
#endif

namespace slm {

// Defined in beam_select.cu
size_t beam_select_workspace_bytes(int W_in, int V, int W);
bool beam_select_supported(int W_in, int V, int W);
cudaError_t launch_beam_select(const void* logits, const float* cum, int W_in, int V, int W, int32_t* out_token,
                               int32_t* out_parent, float* out_score, int32_t* out_cand_token,
                               int32_t* out_cand_parent, float* out_cand_score, float* out_lse, void* workspace,
                               cudaStream_t stream);

// Defined in heads.cu
cudaError_t launch_swiglu_quant(const void* gate_up, int T, int I, void* q, float* scale, int num_sms,
                                cudaStream_t stream);
cudaError_t launch_label_scores(const void* hidden, const int32_t* cu, int B, int T, int d, const void* w_label,
                                int n_labels, float* logits, float* probs, int32_t* dev_status, cudaStream_t stream);
cudaError_t launch_beam_finished(const int32_t* cand_token, const int32_t* cand_parent, const float* cand_score, int W,
                                 int stop_id, int32_t* out_token, int32_t* out_parent, float* out_score,
                                 int32_t* fin_token, int32_t* fin_parent, float* fin_score, int32_t* fin_count,
                                 cudaStream_t stream);
cudaError_t launch_beam_history(const int32_t* hist_in, const int32_t* parent, const int32_t* token, int W, int W_in,
                                int t, int max_len, int32_t* hist_out, int32_t* dev_status, cudaStream_t stream);

namespace {

thread_local std::string g_last_error;

slm_status fail(slm_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

slm_status ok() {
  g_last_error.clear();
  return SLM_OK;
}

slm_status cuda_fail(cudaError_t e, const char* what) {
  return fail(SLM_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Limit of every bounded wait inside the attention kernels, read when a call
// fills its launch parameters (slm_set_wait_timeout_ns).
std::atomic<uint64_t> g_wait_ns{kWaitTimeoutNs};

// ---- TMA descriptor encoding through the driver entry point ----------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiledFn>(nullptr);
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// bf16 tensor [d2, d1, d0] (d0 contiguous), 128-byte swizzled boxes
// {64, box1, box2}; out-of-range elements read as zero.
bool encode_bf16_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t box1,
                    uint32_t box2) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  cuuint32_t box[3] = {64, box1, box2};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  static int cache[64] = {0};
  if (dev < 64 && cache[dev]) return cache[dev];
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  if (dev < 64) cache[dev] = n;
  return n;
}

// Persistent launch: one CTA per SM (or per unit when there are fewer).
template <int D, AttnMode MODE>
cudaError_t launch_attn(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& to,
                        const AttnParams& p, int64_t max_units, cudaStream_t stream) {
  auto kern = p.o_f32 ? attn_fwd_kernel<D, MODE, true> : attn_fwd_kernel<D, MODE, false>;
  const int smem = FwdSmem<D, MODE>::kAlloc;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(num_sms(), max_units)));
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kFwdThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  // a programmatic dependent of the kernel before it (prefill: the schedule
  // kernel launched just before); the kernel waits before reading memory
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, to, p);
}

// ---- prefill tile schedule -------------------------------------------------
constexpr int kSchedThreads = 1024;
constexpr int kMaxKvBlocks = 4095;  // longest sequence: 4095 * 128 tokens
constexpr int kBuckets = 4096;

// Lists the (start, length, pair of query tiles) work items after checking the
// boundary: sequences by length, longest first, and inside a sequence the
// pairs that read the most key blocks first.  Persistent CTAs take the items
// round-robin, so the items of one sequence run at the same time on
// different SMs and share its K/V through L2, and the short ones come last.
__global__ void __launch_bounds__(kSchedThreads)
    prefill_schedule_kernel(const int32_t* cu, int B, int T, int tok2, int max_nb, int32_t* items, int64_t cap,
                            int32_t* dev_status) {
  __shared__ int cnt[kBuckets];
  __shared__ int warp_tot[kSchedThreads / 32];
  __shared__ int bad;
  pdl_launch_dependents();  // the attention kernel may start its setup now
  // the first kSchedThreads sequences' boundaries, loaded once
  const int b_own = threadIdx.x;
  const int s0_own = (b_own < B) ? cu[b_own] : 0;
  const int len_own = (b_own < B) ? cu[b_own + 1] - s0_own : 0;
  auto seq = [&](int b, int& s0, int& len) {
    if (b == b_own) {
      s0 = s0_own;
      len = len_own;
    } else {
      s0 = cu[b];
      len = cu[b + 1] - s0;
    }
  };
  for (int i = threadIdx.x; i < kBuckets; i += kSchedThreads) cnt[i] = 0;
  if (threadIdx.x == 0) bad = (cu[0] != 0 || cu[B] != T) ? 1 : 0;
  __syncthreads();
  for (int b = threadIdx.x; b < B; b += kSchedThreads) {
    int s0, len;
    seq(b, s0, len);
    if (len < 0 || (len + kBlockN - 1) / kBlockN > max_nb) bad = 1;
  }
  __syncthreads();
  if (bad) {
    if (threadIdx.x == 0) {
      items[0] = 0;
      if (dev_status) atomicOr(dev_status, kDevBadSeqlens);
    }
    return;
  }
  for (int b = threadIdx.x; b < B; b += kSchedThreads) {
    int s0, len;
    seq(b, s0, len);
    if (len > 0) atomicAdd(&cnt[(len + kBlockN - 1) / kBlockN], (len + tok2 - 1) / tok2);
  }
  __syncthreads();
  // exclusive scan from the longest bucket down: 4 buckets per thread
  int loc[4], sum = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    loc[i] = cnt[kBuckets - 1 - (4 * threadIdx.x + i)];
    sum += loc[i];
  }
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int x = sum;
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[w] = x;
  __syncthreads();
  int base = 0, total = 0;
  for (int i = 0; i < kSchedThreads / 32; ++i) {
    if (i < w) base += warp_tot[i];
    total += warp_tot[i];
  }
  int run = base + x - sum;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    cnt[kBuckets - 1 - (4 * threadIdx.x + i)] = run;
    run += loc[i];
  }
  __syncthreads();
  for (int b = threadIdx.x; b < B; b += kSchedThreads) {
    int s0, len;
    seq(b, s0, len);
    if (len <= 0) continue;
    const int n_items = (len + tok2 - 1) / tok2;
    const int pos = atomicAdd(&cnt[(len + kBlockN - 1) / kBlockN], n_items);
    for (int k = 0; k < n_items; ++k) {
      if (!in_bounds(pos + k < cap, dev_status)) break;
      items[1 + 3 * (pos + k)] = s0;
      items[2 + 3 * (pos + k)] = len;
      items[3 + 3 * (pos + k)] = n_items - 1 - k;
    }
  }
  if (threadIdx.x == 0) items[0] = total;
}

// Upper bound of the work items: sum over sequences of ceil(L / (2 TOK)).
int64_t prefill_item_capacity(int32_t num_seqs, int32_t total_tokens, int32_t tok) {
  return static_cast<int64_t>(total_tokens) / (2 * tok) + num_seqs + 1;
}

}  // namespace
}  // namespace slm

using namespace slm;

extern "C" {

const char* slm_last_error(void) { return g_last_error.c_str(); }

int32_t slm_abi_version(void) { return 2; }

size_t slm_prefill_workspace_size(int32_t num_seqs, int32_t total_tokens, int32_t max_seqlen, int32_t n_q_heads,
                                  int32_t n_kv_heads) {
  (void)max_seqlen;
  if (num_seqs < 0 || total_tokens < 0 || n_q_heads <= 0 || n_kv_heads <= 0 || n_q_heads % n_kv_heads) return 0;
  const int G = n_q_heads / n_kv_heads;
  if (G > kBlockM) return 0;
  const int64_t cap = prefill_item_capacity(num_seqs, total_tokens, kBlockM / G);
  return static_cast<size_t>(((1 + 3 * cap) * 4 + 255) / 256 * 256);
}

}  // extern "C"

namespace {

// Packed prefill with a bf16 output o, or (o_f32 non-null) an fp32 one.
slm_status prefill_impl(const void* q, const void* k, const void* v, const int32_t* cu_seqlens,
                        const int32_t* cu_seqlens_host, int32_t num_seqs, int32_t total_tokens, int32_t max_seqlen,
                        int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim, float softmax_scale, void* o_bf16,
                        float* o_f32, float* lse, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                        void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  void* o = o_f32 ? static_cast<void*>(o_f32) : o_bf16;
  if (num_seqs < 0 || total_tokens < 0 || max_seqlen < 0)
    return fail(SLM_ERR_INVALID_ARG, "negative size (num_seqs=%d total_tokens=%d max_seqlen=%d)", num_seqs,
                total_tokens, max_seqlen);
  if (n_q_heads <= 0 || n_kv_heads <= 0 || n_q_heads % n_kv_heads != 0)
    return fail(SLM_ERR_INVALID_ARG, "need n_q_heads %% n_kv_heads == 0 (got %d, %d)", n_q_heads, n_kv_heads);
  if (head_dim != 64 && head_dim != 128)
    return fail(SLM_ERR_UNSUPPORTED, "head_dim %d unsupported (64 or 128)", head_dim);
  const int G = n_q_heads / n_kv_heads;
  if (G > kBlockM) return fail(SLM_ERR_UNSUPPORTED, "query heads per KV head %d > %d", G, kBlockM);
  if (!(softmax_scale > 0.f) || !std::isfinite(softmax_scale))
    return fail(SLM_ERR_INVALID_ARG, "softmax_scale must be finite and > 0");
  if ((max_seqlen + kBlockN - 1) / kBlockN > kMaxKvBlocks)
    return fail(SLM_ERR_UNSUPPORTED, "max_seqlen %d above %d", max_seqlen, kMaxKvBlocks * kBlockN);
  if (cu_seqlens_host) {
    if (cu_seqlens_host[0] != 0 || cu_seqlens_host[num_seqs] != total_tokens)
      return fail(SLM_ERR_INVALID_ARG, "cu_seqlens must start at 0 and end at total_tokens");
    for (int b = 0; b < num_seqs; ++b) {
      const int len = cu_seqlens_host[b + 1] - cu_seqlens_host[b];
      if (len < 0) return fail(SLM_ERR_INVALID_ARG, "cu_seqlens decreases at %d", b);
      if (len > max_seqlen) return fail(SLM_ERR_INVALID_ARG, "sequence %d longer than max_seqlen", b);
    }
  }
  if (total_tokens == 0) return ok();
  if (!q || !k || !v || !o || !cu_seqlens)
    return fail(SLM_ERR_INVALID_ARG, "null q/k/v/o/cu_seqlens");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
    return fail(SLM_ERR_INVALID_ARG, "q/k/v/o must be 16-byte aligned");
  if (o == q || o == k || o == v) return fail(SLM_ERR_INVALID_ARG, "o aliases an input");
  const size_t need = slm_prefill_workspace_size(num_seqs, total_tokens, max_seqlen, n_q_heads, n_kv_heads);
  if (!workspace || workspace_bytes < need)
    return fail(SLM_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", workspace ? workspace_bytes : 0, need);
  if (!aligned16(workspace)) return fail(SLM_ERR_INVALID_ARG, "workspace must be 16-byte aligned");

  const int tok = kBlockM / G;
  const int64_t cap = prefill_item_capacity(num_seqs, total_tokens, tok);
  if (cap * n_kv_heads > 0x7FFFFFFF) return fail(SLM_ERR_UNSUPPORTED, "too many tiles");
  // A softmax warp's 32 rows are whole tokens when G divides 32: those warps
  // write their rows through a {64, G, 32 / G} box of the output map.
  const bool warp_tma_store = (o_f32 == nullptr) && (32 % G == 0);
  CUtensorMap tq, tk, tv, to;
  if (!encode_bf16_3d(&tq, q, head_dim, n_q_heads, total_tokens, G, tok) ||
      !encode_bf16_3d(&tk, k, head_dim, n_kv_heads, total_tokens, 1, kBlockN) ||
      !encode_bf16_3d(&tv, v, head_dim, n_kv_heads, total_tokens, 1, kBlockN))
    return fail(SLM_ERR_CUDA, "cuTensorMapEncodeTiled failed");
  if (warp_tma_store) {
    if (!encode_bf16_3d(&to, o, head_dim, n_q_heads, total_tokens, G, 32 / G))
      return fail(SLM_ERR_CUDA, "cuTensorMapEncodeTiled failed (o)");
  } else {
    to = tq;  // not used
  }

  int32_t* items = static_cast<int32_t*>(workspace);
  const int max_nb = std::max(1, (max_seqlen + kBlockN - 1) / kBlockN);
  prefill_schedule_kernel<<<1, kSchedThreads, 0, stream>>>(cu_seqlens, num_seqs, total_tokens, 2 * tok, max_nb,
                                                           items, cap, dev_status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "prefill schedule launch");

  AttnParams p{};
  p.n_q_heads = n_q_heads;
  p.n_kv_heads = n_kv_heads;
  p.group = G;
  p.tok_per_tile = tok;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  p.o = static_cast<__nv_bfloat16*>(o_bf16);
  p.o_f32 = o_f32;
  p.lse = lse;
  p.dev_status = dev_status;
  p.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
  p.warp_tma_store = warp_tma_store ? 1 : 0;
  p.cu_seqlens = cu_seqlens;
  p.items = items;
  p.items_cap = static_cast<int>(cap);
  p.total_tokens = total_tokens;
  e = (head_dim == 64) ? launch_attn<64, AttnMode::kPrefill>(tq, tk, tv, to, p, cap * n_kv_heads, stream)
                       : launch_attn<128, AttnMode::kPrefill>(tq, tk, tv, to, p, cap * n_kv_heads, stream);
  if (e != cudaSuccess) return cuda_fail(e, "prefill attention launch");
  return ok();
}

}  // namespace

extern "C" {

slm_status slm_packed_prefill_attn(const void* q, const void* k, const void* v, const int32_t* cu_seqlens,
                                   const int32_t* cu_seqlens_host, int32_t num_seqs, int32_t total_tokens,
                                   int32_t max_seqlen, int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
                                   float softmax_scale, void* o, float* lse, void* workspace, size_t workspace_bytes,
                                   int32_t* dev_status, void* stream) {
  SLM_RANGE("slm_packed_prefill_attn");
  return prefill_impl(q, k, v, cu_seqlens, cu_seqlens_host, num_seqs, total_tokens, max_seqlen, n_q_heads,
                      n_kv_heads, head_dim, softmax_scale, o, nullptr, lse, workspace, workspace_bytes, dev_status,
                      stream);
}

slm_status slm_packed_prefill_attn_f32(const void* q, const void* k, const void* v, const int32_t* cu_seqlens,
                                       const int32_t* cu_seqlens_host, int32_t num_seqs, int32_t total_tokens,
                                       int32_t max_seqlen, int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
                                       float softmax_scale, float* o, float* lse, void* workspace,
                                       size_t workspace_bytes, int32_t* dev_status, void* stream) {
  SLM_RANGE("slm_packed_prefill_attn_f32");
  if (total_tokens > 0 && !o) return fail(SLM_ERR_INVALID_ARG, "null o");
  return prefill_impl(q, k, v, cu_seqlens, cu_seqlens_host, num_seqs, total_tokens, max_seqlen, n_q_heads,
                      n_kv_heads, head_dim, softmax_scale, nullptr, o, lse, workspace, workspace_bytes, dev_status,
                      stream);
}

uint64_t slm_set_wait_timeout_ns(uint64_t ns) { return g_wait_ns.exchange(ns); }

// Decode key-split workspace: a fixed area of tickets first (one per beam
// tile pair, KV head, sub-tile and softmax warp; the same place whatever the call's sizes,
// so no call's parts ever land on them), then the split parts of every output
// row (fp32 O and (max, sum)), stored per sub-tile with rows innermost.  The
// tickets must be zero before a call; a call that completes leaves them zero.
constexpr int64_t kMaxDecodeSplit = 16;
constexpr size_t kDecodeTickets = 16384;  // one per warp of every sub-tile
struct DecodeSplitLayout {
  size_t o_off, ml_off, ticket_off, total;
  bool fits;  // the call's tickets fit the fixed area
};
static DecodeSplitLayout decode_split_layout(int n_split, int W, int n_q_heads, int n_kv_heads, int head_dim) {
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  const int tok = kBlockM / (n_q_heads / n_kv_heads);
  const size_t tiles = static_cast<size_t>((W + 2 * tok - 1) / (2 * tok));
  const size_t sub_tiles = tiles * n_kv_heads * 2;
  DecodeSplitLayout l;
  l.ticket_off = 0;
  l.o_off = kDecodeTickets * sizeof(int32_t);
  l.ml_off = l.o_off + up(static_cast<size_t>(n_split) * sub_tiles * kBlockM * head_dim * sizeof(float));
  l.total = l.ml_off + up(static_cast<size_t>(n_split) * sub_tiles * kBlockM * 2 * sizeof(float));
  l.fits = sub_tiles * 4 <= kDecodeTickets;
  return l;
}

}  // extern "C"

namespace {

// Shared-prefix decode with a bf16 output o, or (o_f32 non-null) an fp32 one.
slm_status decode_impl(const void* q, const void* kp, const void* vp, const void* ks, const void* vs,
                       const void* k_new, const void* v_new, const int32_t* parent_idx, int32_t W, int32_t Lp,
                       int32_t L_prev, int32_t Smax, int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
                       float softmax_scale, void* ks_out, void* vs_out, void* o_bf16, float* o_f32, float* lse,
                       int32_t* dev_status, void* workspace, size_t workspace_bytes, void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  void* o = o_f32 ? static_cast<void*>(o_f32) : o_bf16;
  if (W < 0 || Lp < 0 || L_prev < 0 || Smax < 0)
    return fail(SLM_ERR_INVALID_ARG, "negative size (W=%d Lp=%d L_prev=%d Smax=%d)", W, Lp, L_prev, Smax);
  if (n_q_heads <= 0 || n_kv_heads <= 0 || n_q_heads % n_kv_heads != 0)
    return fail(SLM_ERR_INVALID_ARG, "need n_q_heads %% n_kv_heads == 0 (got %d, %d)", n_q_heads, n_kv_heads);
  if (head_dim != 64 && head_dim != 128)
    return fail(SLM_ERR_UNSUPPORTED, "head_dim %d unsupported (64 or 128)", head_dim);
  const int G = n_q_heads / n_kv_heads;
  if (G > kBlockM) return fail(SLM_ERR_UNSUPPORTED, "query heads per KV head %d > %d", G, kBlockM);
  if (!(softmax_scale > 0.f) || !std::isfinite(softmax_scale))
    return fail(SLM_ERR_INVALID_ARG, "softmax_scale must be finite and > 0");
  if ((k_new == nullptr) != (v_new == nullptr)) return fail(SLM_ERR_INVALID_ARG, "k_new and v_new: both or neither");
  const int Ls = L_prev + (k_new ? 1 : 0);
  if (Ls > Smax) return fail(SLM_ERR_INVALID_ARG, "suffix length %d exceeds Smax %d", Ls, Smax);
  if (Lp + Ls < 1) return fail(SLM_ERR_INVALID_ARG, "no keys: Lp + L_s must be >= 1");
  if (W == 0) return ok();
  if (!q || !o) return fail(SLM_ERR_INVALID_ARG, "null q/o");
  if (Lp > 0 && (!kp || !vp)) return fail(SLM_ERR_INVALID_ARG, "null kp/vp with Lp > 0");
  if (L_prev > 0 && (!ks || !vs)) return fail(SLM_ERR_INVALID_ARG, "null ks/vs with L_prev > 0");
  if (Ls > 0 && (!ks_out || !vs_out)) return fail(SLM_ERR_INVALID_ARG, "null ks_out/vs_out");
  const void* ptrs[] = {q, kp, vp, ks, vs, k_new, v_new, ks_out, vs_out, o};
  for (const void* ptr : ptrs)
    if (ptr && !aligned16(ptr)) return fail(SLM_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  if (ks_out && (ks_out == ks || ks_out == vs || vs_out == ks || vs_out == vs || ks_out == vs_out))
    return fail(SLM_ERR_INVALID_ARG, "ks_out/vs_out must not alias ks/vs or each other");
  if (o == q) return fail(SLM_ERR_INVALID_ARG, "o aliases q");

  const int tok = kBlockM / G;
  const int64_t tiles = (W + 2 * tok - 1) / (2 * tok);
  // Split the prompt's key blocks over CTAs when the tiles alone leave most
  // SMs idle and the workspace has room for the split parts.
  const int nb_all = (Lp + kBlockN - 1) / kBlockN;
  int n_split = 1, blk_per_split = nb_all;
  DecodeSplitLayout lay{};
  if (workspace && nb_all > 1) {
    const int64_t base = tiles * n_kv_heads;
    const int want = static_cast<int>(std::min<int64_t>({static_cast<int64_t>(nb_all), kMaxDecodeSplit,
                                                         std::max<int64_t>(1, num_sms() / base)}));
    if (want > 1) {
      const int bps = (nb_all + want - 1) / want;
      const int ns = (nb_all + bps - 1) / bps;
      lay = decode_split_layout(ns, W, n_q_heads, n_kv_heads, head_dim);
      if (lay.fits && aligned16(workspace) && lay.total <= workspace_bytes) {
        n_split = ns;
        blk_per_split = bps;
      }
    }
  }
  const int64_t n_units = tiles * n_kv_heads * n_split;
  CUtensorMap tq, tk, tv;
  std::memset(&tk, 0, sizeof tk);
  std::memset(&tv, 0, sizeof tv);
  if (!encode_bf16_3d(&tq, q, head_dim, n_q_heads, W, G, tok))
    return fail(SLM_ERR_CUDA, "cuTensorMapEncodeTiled failed (q)");
  if (Lp > 0 && (!encode_bf16_3d(&tk, kp, head_dim, n_kv_heads, Lp, 1, kBlockN) ||
                 !encode_bf16_3d(&tv, vp, head_dim, n_kv_heads, Lp, 1, kBlockN)))
    return fail(SLM_ERR_CUDA, "cuTensorMapEncodeTiled failed (prefix)");

  AttnParams p{};
  p.n_q_heads = n_q_heads;
  p.n_kv_heads = n_kv_heads;
  p.group = G;
  p.tok_per_tile = tok;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  p.o = static_cast<__nv_bfloat16*>(o_bf16);
  p.o_f32 = o_f32;
  p.lse = lse;
  p.dev_status = dev_status;
  p.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.ks = static_cast<const __nv_bfloat16*>(ks);
  p.vs = static_cast<const __nv_bfloat16*>(vs);
  p.k_new = static_cast<const __nv_bfloat16*>(k_new);
  p.v_new = static_cast<const __nv_bfloat16*>(v_new);
  p.parent = parent_idx;
  p.ks_out = static_cast<__nv_bfloat16*>(ks_out);
  p.vs_out = static_cast<__nv_bfloat16*>(vs_out);
  p.W = W;
  p.Lp = Lp;
  p.L_prev = L_prev;
  p.Smax = Smax;
  p.n_split = n_split;
  p.blk_per_split = blk_per_split;
  if (n_split > 1) {
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    p.ws_o = reinterpret_cast<float*>(ws + lay.o_off);
    p.ws_ml = reinterpret_cast<float2*>(ws + lay.ml_off);
    p.tickets = reinterpret_cast<int32_t*>(ws + lay.ticket_off);
    p.ws_o_elems = static_cast<int64_t>((lay.ml_off - lay.o_off) / sizeof(float));
    p.tickets_cap = static_cast<int>(kDecodeTickets);
  }
  // decode writes O row by row (the suffix merge ends in registers); the
  // output map argument is unused
  cudaError_t e = (head_dim == 64) ? launch_attn<64, AttnMode::kDecodePrefix>(tq, tk, tv, tq, p, n_units, stream)
                                   : launch_attn<128, AttnMode::kDecodePrefix>(tq, tk, tv, tq, p, n_units, stream);
  if (e != cudaSuccess) return cuda_fail(e, "decode attention launch");
  return ok();
}

}  // namespace

extern "C" {

slm_status slm_shared_prefix_decode_attn(const void* q, const void* kp, const void* vp, const void* ks,
                                         const void* vs, const void* k_new, const void* v_new,
                                         const int32_t* parent_idx, int32_t W, int32_t Lp, int32_t L_prev,
                                         int32_t Smax, int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
                                         float softmax_scale, void* ks_out, void* vs_out, void* o, float* lse,
                                         int32_t* dev_status, void* workspace, size_t workspace_bytes,
                                         void* stream) {
  SLM_RANGE("slm_shared_prefix_decode_attn");
  return decode_impl(q, kp, vp, ks, vs, k_new, v_new, parent_idx, W, Lp, L_prev, Smax, n_q_heads, n_kv_heads,
                     head_dim, softmax_scale, ks_out, vs_out, o, nullptr, lse, dev_status, workspace,
                     workspace_bytes, stream);
}

slm_status slm_shared_prefix_decode_attn_f32(const void* q, const void* kp, const void* vp, const void* ks,
                                             const void* vs, const void* k_new, const void* v_new,
                                             const int32_t* parent_idx, int32_t W, int32_t Lp, int32_t L_prev,
                                             int32_t Smax, int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
                                             float softmax_scale, void* ks_out, void* vs_out, float* o, float* lse,
                                             int32_t* dev_status, void* workspace, size_t workspace_bytes,
                                             void* stream) {
  SLM_RANGE("slm_shared_prefix_decode_attn_f32");
  if (W > 0 && !o) return fail(SLM_ERR_INVALID_ARG, "null o");
  return decode_impl(q, kp, vp, ks, vs, k_new, v_new, parent_idx, W, Lp, L_prev, Smax, n_q_heads, n_kv_heads,
                     head_dim, softmax_scale, ks_out, vs_out, nullptr, o, lse, dev_status, workspace,
                     workspace_bytes, stream);
}

size_t slm_shared_prefix_decode_workspace_size(int32_t W, int32_t Lp, int32_t n_q_heads, int32_t n_kv_heads,
                                              int32_t head_dim) {
  if (W <= 0 || Lp <= 0 || n_q_heads <= 0 || n_kv_heads <= 0 || n_q_heads % n_kv_heads != 0) return 0;
  if (head_dim != 64 && head_dim != 128) return 0;
  const int nb_all = (Lp + kBlockN - 1) / kBlockN;
  if (nb_all <= 1) return 0;
  const int ns = static_cast<int>(std::min<int64_t>(nb_all, kMaxDecodeSplit));
  return decode_split_layout(ns, W, n_q_heads, n_kv_heads, head_dim).total;
}

size_t slm_beam_select_workspace_size(int32_t W_in, int32_t V, int32_t W) {
  if (W_in <= 0 || V <= 0 || W <= 0 || static_cast<int64_t>(2) * W > V) return 0;
  if (!beam_select_supported(W_in, V, W)) return 0;
  return beam_select_workspace_bytes(W_in, V, W);
}

slm_status slm_beam_select(const void* logits, const float* cum_scores, int32_t W_in, int32_t V, int32_t W,
                           int32_t* out_token, int32_t* out_parent, float* out_score, int32_t* out_cand_token,
                           int32_t* out_cand_parent, float* out_cand_score, float* out_lse, void* workspace,
                           size_t workspace_bytes, void* stream_) {
  SLM_RANGE("slm_beam_select");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (W_in <= 0 || V <= 0 || W <= 0)
    return fail(SLM_ERR_INVALID_ARG, "sizes must be positive (W_in=%d V=%d W=%d)", W_in, V, W);
  if (static_cast<int64_t>(2) * W > V) return fail(SLM_ERR_INVALID_ARG, "need 2W <= V (W=%d V=%d)", W, V);
  if (!beam_select_supported(W_in, V, W))
    return fail(SLM_ERR_UNSUPPORTED, "beam sizes W_in=%d W=%d V=%d unsupported", W_in, W, V);
  if (!logits || !cum_scores || !out_token || !out_parent || !out_score)
    return fail(SLM_ERR_INVALID_ARG, "null logits/cum_scores/outputs");
  if (!aligned16(logits)) return fail(SLM_ERR_INVALID_ARG, "logits must be 16-byte aligned");
  const size_t need = beam_select_workspace_bytes(W_in, V, W);
  if (!workspace || workspace_bytes < need)
    return fail(SLM_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", workspace ? workspace_bytes : 0, need);
  if (!aligned16(workspace)) return fail(SLM_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
  cudaError_t e = launch_beam_select(logits, cum_scores, W_in, V, W, out_token, out_parent, out_score,
                                     out_cand_token, out_cand_parent, out_cand_score, out_lse, workspace, stream);
  if (e != cudaSuccess) return cuda_fail(e, "beam select launch");
  return ok();
}

slm_status slm_swiglu_quant_e4m3(const void* gate_up, int32_t T, int32_t I, void* q, float* scale, void* stream_) {
  SLM_RANGE("slm_swiglu_quant_e4m3");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (T < 0 || I <= 0) return fail(SLM_ERR_INVALID_ARG, "need T >= 0 and I > 0 (T=%d I=%d)", T, I);
  if (I % 8 != 0) return fail(SLM_ERR_UNSUPPORTED, "I=%d must be a multiple of 8", I);
  if (T == 0) return ok();
  if (!gate_up || !q || !scale) return fail(SLM_ERR_INVALID_ARG, "null gate_up/q/scale");
  if (!aligned16(gate_up) || !aligned16(q) || !aligned16(scale))
    return fail(SLM_ERR_INVALID_ARG, "gate_up/q/scale must be 16-byte aligned");
  cudaError_t e = launch_swiglu_quant(gate_up, T, I, q, scale, num_sms(), stream);
  if (e != cudaSuccess) return cuda_fail(e, "swiglu quant launch");
  return ok();
}

slm_status slm_label_scores(const void* hidden, const int32_t* cu_seqlens, int32_t num_seqs, int32_t total_tokens,
                            int32_t d_model, const void* w_label, int32_t n_labels, float* logits, float* probs,
                            int32_t* dev_status, void* stream_) {
  SLM_RANGE("slm_label_scores");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (num_seqs < 0 || total_tokens < 0 || d_model <= 0)
    return fail(SLM_ERR_INVALID_ARG, "bad sizes (num_seqs=%d total_tokens=%d d_model=%d)", num_seqs, total_tokens,
                d_model);
  if (n_labels < 1 || n_labels > 32) return fail(SLM_ERR_UNSUPPORTED, "n_labels=%d outside [1, 32]", n_labels);
  if (d_model % 8 != 0) return fail(SLM_ERR_UNSUPPORTED, "d_model=%d must be a multiple of 8", d_model);
  if (num_seqs == 0) return ok();
  if (!hidden || !cu_seqlens || !w_label || !logits) return fail(SLM_ERR_INVALID_ARG, "null hidden/cu_seqlens/w_label/logits");
  if (!aligned16(hidden) || !aligned16(w_label)) return fail(SLM_ERR_INVALID_ARG, "hidden/w_label must be 16-byte aligned");
  cudaError_t e = launch_label_scores(hidden, cu_seqlens, num_seqs, total_tokens, d_model, w_label, n_labels, logits,
                                      probs, dev_status, stream);
  if (e != cudaSuccess) return cuda_fail(e, "label scores launch");
  return ok();
}

slm_status slm_beam_split_finished(const int32_t* cand_token, const int32_t* cand_parent, const float* cand_score,
                                   int32_t W, int32_t stop_id, int32_t* out_token, int32_t* out_parent,
                                   float* out_score, int32_t* fin_token, int32_t* fin_parent, float* fin_score,
                                   int32_t* fin_count, void* stream_) {
  SLM_RANGE("slm_beam_split_finished");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (W < 1 || W > 1024) return fail(SLM_ERR_INVALID_ARG, "W=%d outside [1, 1024]", W);
  if (!cand_token || !cand_parent || !cand_score || !out_token || !out_parent || !out_score || !fin_token ||
      !fin_parent || !fin_score || !fin_count)
    return fail(SLM_ERR_INVALID_ARG, "null pointer argument");
  cudaError_t e = launch_beam_finished(cand_token, cand_parent, cand_score, W, stop_id, out_token, out_parent, out_score,
                                       fin_token, fin_parent, fin_score, fin_count, stream);
  if (e != cudaSuccess) return cuda_fail(e, "finished split launch");
  return ok();
}

slm_status slm_beam_reorder_history(const int32_t* hist_in, const int32_t* parent_idx, const int32_t* token,
                                    int32_t W, int32_t W_in, int32_t t, int32_t max_len, int32_t* hist_out,
                                    int32_t* dev_status, void* stream_) {
  SLM_RANGE("slm_beam_reorder_history");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (W < 1 || W_in < 1 || t < 0 || max_len < 1 || t >= max_len)
    return fail(SLM_ERR_INVALID_ARG, "bad sizes (W=%d W_in=%d t=%d max_len=%d)", W, W_in, t, max_len);
  if (!token || !hist_out || (t > 0 && !hist_in)) return fail(SLM_ERR_INVALID_ARG, "null token/hist_out/hist_in");
  if (hist_in == hist_out) return fail(SLM_ERR_INVALID_ARG, "hist_out aliases hist_in");
  cudaError_t e = launch_beam_history(hist_in, parent_idx, token, W, W_in, t, max_len, hist_out, dev_status, stream);
  if (e != cudaSuccess) return cuda_fail(e, "history reorder launch");
  return ok();
}

slm_status slm_check_status(const int32_t* dev_status, void* stream_) {
  if (!dev_status) return fail(SLM_ERR_INVALID_ARG, "null dev_status");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  int32_t h = 0;
  cudaError_t e = cudaMemcpyAsync(&h, dev_status, sizeof h, cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "reading dev_status");
  if (h != 0)
    return fail(SLM_ERR_DEVICE_CHECK, "device status 0x%x:%s%s%s%s", h, (h & kDevBadSeqlens) ? " bad-cu_seqlens" : "",
                (h & kDevBadParent) ? " bad-parent-index" : "", (h & kDevPipelineTimeout) ? " pipeline-timeout" : "",
                (h & kDevBounds) ? " index-out-of-bounds" : "");
  return ok();
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Prefill without a caller workspace.
//
// Some callers cannot allocate device memory at the point where they run
// attention: code inside a frozen, ahead-of-time compiled graph whose memory
// plan is fixed, a runtime whose only allocator is busy or forbidden on the
// hot path, or a plugin host that hands out inputs and outputs but no scratch.
// For them the tile schedule lives in a fixed array of this library's own
// device memory, created when the library is loaded on a GPU and held until
// the process exits.
// ---------------------------------------------------------------------------
namespace {

// Work items the array holds: one int32 count plus (start, length, pair)
// per item, 192 KiB in total.
constexpr int64_t kNoAllocMaxItems = 16383;
constexpr int64_t kNoAllocInts = 1 + 3 * kNoAllocMaxItems + 2;  // padded to 256-byte multiple
static __device__ __align__(256) int32_t g_noalloc_items[kNoAllocInts];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_addr[kMaxDevices] = {nullptr};

// Device address of the array on the current device, looked up once per
// device (host code only ever sees a stand-in for the symbol).
slm_status noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(SLM_ERR_UNSUPPORTED, "device ordinal %d above %d", dev, kMaxDevices);
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_addr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_items);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress of the built-in prefill schedule buffer");
    g_noalloc_addr[dev] = ptr;
  }
  *out = g_noalloc_addr[dev];
  return SLM_OK;
}

}  // namespace

extern "C" slm_status slm_packed_prefill_attn_noalloc(const void* q, const void* k, const void* v,
                                                       const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                                                       int32_t num_seqs, int32_t total_tokens, int32_t max_seqlen,
                                                       int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
                                                       float softmax_scale, void* o, float* lse, int32_t* dev_status,
                                                       void* stream) {
  SLM_RANGE("slm_packed_prefill_attn_noalloc");
  if (num_seqs < 0 || total_tokens < 0 || n_q_heads <= 0 || n_kv_heads <= 0 || n_q_heads % n_kv_heads != 0)
    return slm_packed_prefill_attn(q, k, v, cu_seqlens, cu_seqlens_host, num_seqs, total_tokens, max_seqlen,
                                   n_q_heads, n_kv_heads, head_dim, softmax_scale, o, lse, nullptr, 0, dev_status,
                                   stream);  // reports the argument error
  const int G = n_q_heads / n_kv_heads;
  if (G <= kBlockM) {
    const int64_t items = prefill_item_capacity(num_seqs, total_tokens, kBlockM / G);
    if (items > kNoAllocMaxItems)
      return fail(SLM_ERR_UNSUPPORTED,
                  "slm_packed_prefill_attn_noalloc: %lld work items exceed its built-in buffer of %lld "
                  "(items = total_tokens / (2 * (128 / (n_q_heads / n_kv_heads))) + num_seqs + 1); "
                  "use slm_packed_prefill_attn with a workspace",
                  static_cast<long long>(items), static_cast<long long>(kNoAllocMaxItems));
  }
  void* scratch = nullptr;
  const slm_status st = noalloc_scratch(&scratch);
  if (st != SLM_OK) return st;
  return slm_packed_prefill_attn(q, k, v, cu_seqlens, cu_seqlens_host, num_seqs, total_tokens, max_seqlen, n_q_heads,
                                 n_kv_heads, head_dim, softmax_scale, o, lse, scratch, sizeof(g_noalloc_items),
                                 dev_status, stream);
}
