// Kernels around the attention hot path (article "SLM 生成式高并发推理引擎：延迟约束下的
// 有效吞吐优化"):
//
//   * fused SwiGLU + per-token dynamic E4M3 re-quantisation (section 3.4): one
//     pass per token row: FP32 SiLU(gate) * up, the row's absolute maximum,
//     its scale, and the E4M3 codes -- no BF16 SwiGLU intermediate;
//   * last-valid-token extraction and label scoring for Prefill-Only models
//     (sections 1.1 and 3.1): each sequence's last row, found through the
//     same sequence boundary as attention, dotted with the label tokens'
//     head rows in FP32, then a softmax over the labels;
//   * finished-beam handling with 2W global candidates (section 3.3):
//     candidates that end in the stop token are set aside, W active beams go
//     on;
//   * the per-step token-history reorder of fixed-depth beam search
//     (section 2.3): each new beam takes its parent's tokens plus its own.
#include <cfloat>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "slm_internal.h"
#include "sm103_ptx.cuh"

namespace slm {
namespace heads {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float warp_max(float v) {
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// ---------------------------------------------------------------------------
// SwiGLU + E4M3
// ---------------------------------------------------------------------------
constexpr int kSwThreads = 256;
constexpr float kE4M3Max = 448.f;  // largest finite E4M3 value

// FP32 SiLU(g) * u: g * sigmoid(g), sigmoid through exp2 and a reciprocal.
__device__ __forceinline__ float swiglu(float g, float u) {
  const float e = exp2f(-g * 1.4426950408889634f);
  return __fdividef(g, 1.f + e) * u;
}

// Two fp32 values -> two E4M3 codes (round to nearest even, saturating to
// +-448), low value in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}

// Row r of gate_up holds gate [I] then up [I].  kVec 16-byte vectors per
// thread and half row stay in registers between the maximum and the codes.
template <int kVec>
__global__ void __launch_bounds__(kSwThreads) swiglu_quant_kernel(const uint16_t* __restrict__ gu, int T, int I,
                                                                  uint8_t* __restrict__ q, float* __restrict__ scale) {
  __shared__ float wmax[kSwThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int nv = I / 8;
  for (int row = blockIdx.x; row < T; row += gridDim.x) {
    const uint4* g4 = reinterpret_cast<const uint4*>(gu + static_cast<int64_t>(row) * 2 * I);
    const uint4* u4 = reinterpret_cast<const uint4*>(gu + static_cast<int64_t>(row) * 2 * I + I);
    uint4 gv[kVec], uv[kVec];
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
      const int v = tid + k * kSwThreads;
      if (v < nv) {
        gv[k] = __ldcs(g4 + v);  // read once: do not keep in cache
        uv[k] = __ldcs(u4 + v);
      }
    }
    float h[kVec][8];
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
      const int v = tid + k * kSwThreads;
      if (v < nv) {
        const uint32_t gw[4] = {gv[k].x, gv[k].y, gv[k].z, gv[k].w};
        const uint32_t uw[4] = {uv[k].x, uv[k].y, uv[k].z, uv[k].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          h[k][2 * e] = swiglu(bf16_lo(gw[e]), bf16_lo(uw[e]));
          h[k][2 * e + 1] = swiglu(bf16_hi(gw[e]), bf16_hi(uw[e]));
          amax = fmaxf(amax, fmaxf(fabsf(h[k][2 * e]), fabsf(h[k][2 * e + 1])));
        }
      }
    }
    amax = warp_max(amax);
    if (lane == 0) wmax[w] = amax;
    __syncthreads();
    amax = wmax[0];
#pragma unroll
    for (int i = 1; i < kSwThreads / 32; ++i) amax = fmaxf(amax, wmax[i]);
    // scale = amax / 448; codes of h * (448 / amax); an all-zero row keeps
    // scale 1 and codes 0
    const float inv = amax > 0.f ? __fdiv_rn(kE4M3Max, amax) : 0.f;
    if (tid == 0) scale[row] = amax > 0.f ? __fdiv_rn(amax, kE4M3Max) : 1.f;
    uint2* q2 = reinterpret_cast<uint2*>(q + static_cast<int64_t>(row) * I);
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
      const int v = tid + k * kSwThreads;
      if (v < nv) {
        uint32_t b[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) b[e] = e4m3x2(h[k][2 * e] * inv, h[k][2 * e + 1] * inv);
        __stcs(q2 + v, make_uint2(b[0] | (b[1] << 16), b[2] | (b[3] << 16)));
      }
    }
    __syncthreads();  // wmax is rewritten by the next row
  }
}

// Rows longer than the register-resident path: the maximum pass, then the
// row read again (from L2) for the codes.
__global__ void __launch_bounds__(kSwThreads) swiglu_quant_long_kernel(const uint16_t* __restrict__ gu, int T, int I,
                                                                       uint8_t* __restrict__ q,
                                                                       float* __restrict__ scale) {
  __shared__ float wmax[kSwThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int nv = I / 8;
  for (int row = blockIdx.x; row < T; row += gridDim.x) {
    const uint4* g4 = reinterpret_cast<const uint4*>(gu + static_cast<int64_t>(row) * 2 * I);
    const uint4* u4 = reinterpret_cast<const uint4*>(gu + static_cast<int64_t>(row) * 2 * I + I);
    float amax = 0.f;
    for (int v = tid; v < nv; v += kSwThreads) {
      const uint4 gv = g4[v], uv = u4[v];
      const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
      const uint32_t uw[4] = {uv.x, uv.y, uv.z, uv.w};
#pragma unroll
      for (int e = 0; e < 4; ++e)
        amax = fmaxf(amax, fmaxf(fabsf(swiglu(bf16_lo(gw[e]), bf16_lo(uw[e]))),
                                 fabsf(swiglu(bf16_hi(gw[e]), bf16_hi(uw[e])))));
    }
    amax = warp_max(amax);
    if (lane == 0) wmax[w] = amax;
    __syncthreads();
    amax = wmax[0];
#pragma unroll
    for (int i = 1; i < kSwThreads / 32; ++i) amax = fmaxf(amax, wmax[i]);
    const float inv = amax > 0.f ? __fdiv_rn(kE4M3Max, amax) : 0.f;
    if (tid == 0) scale[row] = amax > 0.f ? __fdiv_rn(amax, kE4M3Max) : 1.f;
    uint2* q2 = reinterpret_cast<uint2*>(q + static_cast<int64_t>(row) * I);
    for (int v = tid; v < nv; v += kSwThreads) {
      const uint4 gv = g4[v], uv = u4[v];
      const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
      const uint32_t uw[4] = {uv.x, uv.y, uv.z, uv.w};
      uint32_t b[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        b[e] = e4m3x2(swiglu(bf16_lo(gw[e]), bf16_lo(uw[e])) * inv, swiglu(bf16_hi(gw[e]), bf16_hi(uw[e])) * inv);
      q2[v] = make_uint2(b[0] | (b[1] << 16), b[2] | (b[3] << 16));
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// Last-token label scores
// ---------------------------------------------------------------------------
constexpr int kLabThreads = 128;
constexpr int kMaxLabels = 32;

// One CTA per sequence: its last row of hidden states against the label
// rows, FP32 dot products, then an FP32 softmax over the labels.
__global__ void __launch_bounds__(kLabThreads) label_scores_kernel(const uint16_t* __restrict__ hidden,
                                                                   const int32_t* __restrict__ cu, int B, int T, int d,
                                                                   const uint16_t* __restrict__ wl, int n_labels,
                                                                   float* __restrict__ logits,
                                                                   float* __restrict__ probs, int32_t* dev_status) {
  __shared__ float part[kLabThreads / 32][kMaxLabels];
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int s0 = cu[b], s1 = cu[b + 1];
  const bool bad = s0 < 0 || s1 > T || s1 < s0;
  if (bad || s1 == s0) {  // no last token: NaN scores (and a flag if malformed)
    if (tid < n_labels) {
      logits[static_cast<int64_t>(b) * n_labels + tid] = __int_as_float(0x7fc00000);
      if (probs) probs[static_cast<int64_t>(b) * n_labels + tid] = __int_as_float(0x7fc00000);
    }
    if (bad && tid == 0 && dev_status) atomicOr(dev_status, kDevBadSeqlens);
    return;
  }
  const uint4* h4 = reinterpret_cast<const uint4*>(hidden + static_cast<int64_t>(s1 - 1) * d);
  float acc[kMaxLabels];
#pragma unroll
  for (int k = 0; k < kMaxLabels; ++k) acc[k] = 0.f;
  for (int v = tid; v < d / 8; v += kLabThreads) {
    const uint4 hv = h4[v];
    const uint32_t hw[4] = {hv.x, hv.y, hv.z, hv.w};
    float hf[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      hf[2 * e] = bf16_lo(hw[e]);
      hf[2 * e + 1] = bf16_hi(hw[e]);
    }
#pragma unroll
    for (int k = 0; k < kMaxLabels; ++k) {
      if (k < n_labels) {
        const uint4 wv = __ldg(reinterpret_cast<const uint4*>(wl + static_cast<int64_t>(k) * d) + v);
        const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          acc[k] = fmaf(hf[2 * e], bf16_lo(ww[e]), acc[k]);
          acc[k] = fmaf(hf[2 * e + 1], bf16_hi(ww[e]), acc[k]);
        }
      }
    }
  }
#pragma unroll
  for (int k = 0; k < kMaxLabels; ++k) {
    if (k < n_labels) {
      const float s = warp_sum(acc[k]);
      if (lane == 0) part[w][k] = s;
    }
  }
  __syncthreads();
  if (w == 0) {
    float z = -INFINITY;
    if (lane < n_labels) {
      z = 0.f;
#pragma unroll
      for (int i = 0; i < kLabThreads / 32; ++i) z += part[i][lane];  // fixed order
      logits[static_cast<int64_t>(b) * n_labels + lane] = z;
    }
    if (probs) {
      const float m = warp_max(z);
      const float e = (lane < n_labels) ? expf(z - m) : 0.f;
      const float s = warp_sum(e);
      if (lane < n_labels) probs[static_cast<int64_t>(b) * n_labels + lane] = e / s;
    }
  }
}

// ---------------------------------------------------------------------------
// Finished beams
// ---------------------------------------------------------------------------
constexpr int kFinThreads = 1024;

// The 2W global candidates in order: those ranked within the first W that
// end in the stop token are finished hypotheses (rank order); the first W
// candidates that do not are the next active beams.
__global__ void __launch_bounds__(kFinThreads) beam_finished_kernel(
    const int32_t* __restrict__ ct, const int32_t* __restrict__ cp, const float* __restrict__ cs, int W, int stop,
    int32_t* __restrict__ at, int32_t* __restrict__ ap, float* __restrict__ as, int32_t* __restrict__ ftok,
    int32_t* __restrict__ fp, float* __restrict__ fs, int32_t* __restrict__ fcount) {
  __shared__ int wa[kFinThreads / 32], wf[kFinThreads / 32];
  __shared__ int carry_a, carry_f;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  if (tid == 0) {
    carry_a = 0;
    carry_f = 0;
  }
  pdl_wait();  // a programmatic dependent of the selection: its results are complete
  pdl_launch_dependents();
  __syncthreads();
  for (int i0 = 0; i0 < 2 * W; i0 += kFinThreads) {
    const int i = i0 + tid;
    const bool valid = i < 2 * W;
    const int tok = valid ? ct[i] : 0;
    const bool is_stop = valid && tok == stop;
    const bool act = valid && !is_stop;
    const bool fin = is_stop && i < W;
    // block exclusive scans of the two flags (thread order = rank order)
    const unsigned ba = __ballot_sync(kFull, act), bf = __ballot_sync(kFull, fin);
    if (lane == 0) {
      wa[w] = __popc(ba);
      wf[w] = __popc(bf);
    }
    __syncthreads();
    int pa = carry_a, pf = carry_f;
    for (int k = 0; k < w; ++k) {
      pa += wa[k];
      pf += wf[k];
    }
    pa += __popc(ba & ((1u << lane) - 1u));
    pf += __popc(bf & ((1u << lane) - 1u));
    if (act && pa < W) {
      at[pa] = tok;
      ap[pa] = cp[i];
      as[pa] = cs[i];
    }
    if (fin) {
      ftok[pf] = tok;
      fp[pf] = cp[i];
      fs[pf] = cs[i];
    }
    __syncthreads();
    if (tid == kFinThreads - 1) {
      int ta = 0, tf = 0;
      for (int k = 0; k < kFinThreads / 32; ++k) {
        ta += wa[k];
        tf += wf[k];
      }
      carry_a += ta;
      carry_f += tf;
    }
    __syncthreads();
  }
  if (tid == 0) *fcount = carry_f;
}

// ---------------------------------------------------------------------------
// Token history reorder
// ---------------------------------------------------------------------------
// hist_out[b, s] = hist_in[parent[b], s] for s < t; hist_out[b, t] = token[b].
__global__ void beam_history_kernel(const int32_t* __restrict__ hin, const int32_t* __restrict__ parent,
                                    const int32_t* __restrict__ token, int W, int W_in, int t, int max_len,
                                    int32_t* __restrict__ hout, int32_t* dev_status) {
  pdl_wait();  // a programmatic dependent of the kernel before it: its outputs are complete
  pdl_launch_dependents();
  const int b = blockIdx.x;
  int src = parent ? parent[b] : b;
  if (t > 0 && (src < 0 || src >= W_in)) {  // at t = 0 no row is gathered
    if (threadIdx.x == 0 && dev_status) atomicOr(dev_status, kDevBadParent);
    src = 0;
  }
  for (int s = threadIdx.x; s <= t; s += blockDim.x)
    hout[static_cast<int64_t>(b) * max_len + s] = (s < t) ? hin[static_cast<int64_t>(src) * max_len + s] : token[b];
}

}  // namespace heads

// ---------------------------------------------------------------------------
// Launchers (argument checks are done by the C ABI in api.cu)
// ---------------------------------------------------------------------------
cudaError_t launch_swiglu_quant(const void* gate_up, int T, int I, void* q, float* scale, int num_sms,
                                cudaStream_t stream) {
  using namespace heads;
  const int grid = T < num_sms * 8 ? T : num_sms * 8;
  const int per = (I / 8 + kSwThreads - 1) / kSwThreads;  // vectors per thread and half row
  const uint16_t* gu = static_cast<const uint16_t*>(gate_up);
  uint8_t* qq = static_cast<uint8_t*>(q);
  if (per <= 1) swiglu_quant_kernel<1><<<grid, kSwThreads, 0, stream>>>(gu, T, I, qq, scale);
  else if (per == 2) swiglu_quant_kernel<2><<<grid, kSwThreads, 0, stream>>>(gu, T, I, qq, scale);
  else if (per == 3) swiglu_quant_kernel<3><<<grid, kSwThreads, 0, stream>>>(gu, T, I, qq, scale);
  else if (per == 4) swiglu_quant_kernel<4><<<grid, kSwThreads, 0, stream>>>(gu, T, I, qq, scale);
  else swiglu_quant_long_kernel<<<grid, kSwThreads, 0, stream>>>(gu, T, I, qq, scale);
  return cudaGetLastError();
}

cudaError_t launch_label_scores(const void* hidden, const int32_t* cu, int B, int T, int d, const void* w_label,
                                int n_labels, float* logits, float* probs, int32_t* dev_status, cudaStream_t stream) {
  using namespace heads;
  label_scores_kernel<<<B, kLabThreads, 0, stream>>>(static_cast<const uint16_t*>(hidden), cu, B, T, d,
                                                     static_cast<const uint16_t*>(w_label), n_labels, logits, probs,
                                                     dev_status);
  return cudaGetLastError();
}

cudaError_t launch_beam_finished(const int32_t* cand_token, const int32_t* cand_parent, const float* cand_score, int W,
                                 int stop_id, int32_t* out_token, int32_t* out_parent, float* out_score,
                                 int32_t* fin_token, int32_t* fin_parent, float* fin_score, int32_t* fin_count,
                                 cudaStream_t stream) {
  using namespace heads;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(attr, dim3(1), dim3(kFinThreads), stream);
  return cudaLaunchKernelEx(&cfg, beam_finished_kernel, cand_token, cand_parent, cand_score, W, stop_id, out_token,
                            out_parent, out_score, fin_token, fin_parent, fin_score, fin_count);
}

cudaError_t launch_beam_history(const int32_t* hist_in, const int32_t* parent, const int32_t* token, int W, int W_in,
                                int t, int max_len, int32_t* hist_out, int32_t* dev_status, cudaStream_t stream) {
  using namespace heads;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(attr, dim3(W), dim3(32), stream);
  return cudaLaunchKernelEx(&cfg, beam_history_kernel, hist_in, parent, token, W, W_in, t, max_len, hist_out,
                            dev_status);
}

}  // namespace slm
