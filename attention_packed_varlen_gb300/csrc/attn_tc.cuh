// Blackwell (sm_103a) attention core shared by packed prefill and the
// shared-prefix decode: 128 query rows per CTA against a stream of 128-key
// blocks, S = Q K^T and O += P V on tcgen05 with accumulators in TMEM,
// operands staged by TMA in 128-byte-swizzled shared memory, online softmax
// in fp32 by four warps that each own 32 TMEM lanes (one query row per thread).
//
// Query rows are (token, head-in-group) pairs: a tile holds TOK = 128 / G
// consecutive tokens (prefill: positions of one sequence; decode: beams) times
// the G query heads that read one KV head, so every K/V block is loaded once
// for the whole head group ("Triton Packed GQA" in section 3.1 of the article
// "SLM 生成式高并发推理引擎：延迟约束下的有效吞吐优化" does not expand K/V heads either).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "sm103_ptx.cuh"
#include "slm_internal.h"

namespace slm {

constexpr int kBlockM = 128;       // query rows per tile (TMEM lanes)
constexpr int kBlockN = 128;       // keys per block
constexpr int kThreads = 192;      // 4 softmax warps + producer warp + MMA warp
constexpr int kSubTileBytes = 128 * 128;  // 128 rows x 64 bf16
constexpr uint32_t kTmemCols = 512;
constexpr float kLazyRescaleLog2 = 8.0f;  // keep the running max unless it grows by > 2^8

enum class AttnMode : int { kPrefill = 0, kDecodePrefix = 1 };

struct AttnParams {
  // shared
  int n_q_heads, n_kv_heads, group, tok_per_tile;
  float scale_log2;          // softmax_scale * log2(e)
  __nv_bfloat16* o;
  float* lse;                // nullable
  int32_t* dev_status;       // nullable
  // prefill
  const int32_t* cu_seqlens;
  const int32_t* tiles;      // [0] = count, then (seq, q_tile) pairs, heaviest first
  int total_tokens;
  // decode
  const __nv_bfloat16* ks;
  const __nv_bfloat16* vs;
  const __nv_bfloat16* k_new;  // nullable (no append)
  const __nv_bfloat16* v_new;
  const int32_t* parent;     // nullable (identity)
  __nv_bfloat16* ks_out;
  __nv_bfloat16* vs_out;
  int W, Lp, L_prev, Smax;
};

template <int D>
struct SmemLayout {
  static constexpr int kDSub = D / 64;                       // 64-column swizzle blocks
  static constexpr int kQBytes = kDSub * kSubTileBytes;      // 128 rows x D
  static constexpr int kKVBytes = kDSub * kSubTileBytes;     // 128 keys x D
  static constexpr int kPBytes = 2 * kSubTileBytes;          // 128 rows x 128 keys
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kQBytes;                    // 2 stages
  static constexpr int kV = kK + 2 * kKVBytes;               // 2 stages
  static constexpr int kP = kV + 2 * kKVBytes;
  static constexpr int kBar = kP + kPBytes;
  static constexpr int kNumBars = 16;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kTotal = kMisc + 64;
  // Room to align the base to 1024 bytes; at least 116 KB so two CTAs never
  // share an SM (each allocates the SM's 512 TMEM columns).
  static constexpr int kAlloc = (kTotal + 1024) > 118784 ? (kTotal + 1024) : 118784;
};

// Barrier slots
enum : int {
  BAR_Q_FULL = 0,
  BAR_K_FULL = 1,   // +stage
  BAR_K_EMPTY = 3,  // +stage
  BAR_V_FULL = 5,   // +stage
  BAR_V_EMPTY = 7,  // +stage
  BAR_S_FULL = 9,   // +buffer
  BAR_S_FREE = 11,  // +buffer
  BAR_P_FULL = 13,
  BAR_O_READY = 14,
  BAR_DRAIN = 15,
};

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  bool ok = mbar_wait(bar, parity, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

template <int D, AttnMode MODE>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const AttnParams p) {
  using L = SmemLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.group;
  const int TOK = p.tok_per_tile;
  const int rows_used = TOK * G;
  // blockIdx.x = tile * Hkv + kv head: the heaviest tiles of every head group
  // are scheduled first.
  const int kvh = static_cast<int>(blockIdx.x) % p.n_kv_heads;
  const int tile = static_cast<int>(blockIdx.x) / p.n_kv_heads;

  // ---- work item ---------------------------------------------------------
  int row0_global;   // prefill: first token of the tile; decode: first beam
  int n_tok_valid;   // valid tokens (beams) in this tile
  int q0_local = 0;  // prefill: position of the tile's first token in its sequence
  int kv_begin;      // first key row (global index into K/V)
  int n_keys;        // keys the tile reads through the tensor core
  if constexpr (MODE == AttnMode::kPrefill) {
    const int n_tiles = p.tiles[0];
    if (tile >= n_tiles) return;
    const int seq = p.tiles[1 + 2 * tile];
    const int qt = p.tiles[2 + 2 * tile];
    const int s0 = p.cu_seqlens[seq];
    const int len = p.cu_seqlens[seq + 1] - s0;
    q0_local = qt * TOK;
    row0_global = s0 + q0_local;
    n_tok_valid = min(TOK, len - q0_local);
    kv_begin = s0;
    n_keys = q0_local + n_tok_valid;  // causal: keys up to the tile's last query
  } else {
    row0_global = tile * TOK;
    if (row0_global >= p.W) return;
    n_tok_valid = min(TOK, p.W - row0_global);
    kv_begin = 0;
    n_keys = p.Lp;
  }
  const int nblk = (n_keys + kBlockN - 1) / kBlockN;

  // ---- setup ---------------------------------------------------------------
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(&bars[BAR_Q_FULL], 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars[BAR_K_FULL + s], 1);
      mbar_init(&bars[BAR_K_EMPTY + s], 1);
      mbar_init(&bars[BAR_V_FULL + s], 1);
      mbar_init(&bars[BAR_V_EMPTY + s], 1);
      mbar_init(&bars[BAR_S_FULL + s], 1);
      mbar_init(&bars[BAR_S_FREE + s], 128);
    }
    mbar_init(&bars[BAR_P_FULL], 128);
    mbar_init(&bars[BAR_O_READY], 1);
    mbar_init(&bars[BAR_DRAIN], 1);
    fence_mbarrier_init();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    if (nblk > 0) {  // the K/V maps are left empty when there is no prefix
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
    }
  }
  // Rows of the Q tile that the TMA box does not cover (G not dividing 128)
  // must hold finite values: zero them.
  if (rows_used < kBlockM) {
    for (int i = threadIdx.x; i < (kBlockM - rows_used) * L::kDSub * 8; i += kThreads) {
      const int chunk = i & 7;
      const int rest = i >> 3;
      const int r = rows_used + rest % (kBlockM - rows_used);
      const int sub = rest / (kBlockM - rows_used);
      uint4* dst = reinterpret_cast<uint4*>(smem + L::kQ + sub * kSubTileBytes + r * 128 + chunk * 16);
      *dst = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t tS0 = tmem_base;           // S buffers: columns [0,128) and [128,256)
  const uint32_t tO = tmem_base + 256;      // O accumulator: columns [256, 256 + D)

  if (warp == 4) {
    // ======================= TMA producer =======================
    // Decode reads the Q tile in the epilogue too, so it loads Q even when the
    // prefix is empty.
    if (lane == 0 && (nblk > 0 || MODE == AttnMode::kDecodePrefix)) {
      const uint32_t q_bytes = static_cast<uint32_t>(L::kDSub) * 64u * G * TOK * 2u;
      mbar_arrive_expect_tx(&bars[BAR_Q_FULL], q_bytes);
      for (int dh = 0; dh < L::kDSub; ++dh)
        tma_load_3d(smem + L::kQ + dh * kSubTileBytes, &tm_q, &bars[BAR_Q_FULL], dh * 64, kvh * G, row0_global);
      int issued_k = 0, issued_v = 0;
      bool ok = true;
      for (int j = 0; j < nblk && ok; ++j) {
        const int st = j & 1;
        if (j >= 2) ok = mbar_wait(&bars[BAR_K_EMPTY + st], ((j >> 1) - 1) & 1, abort_flag);
        if (!ok) break;
        mbar_arrive_expect_tx(&bars[BAR_K_FULL + st], L::kKVBytes);
        for (int dh = 0; dh < L::kDSub; ++dh)
          tma_load_3d(smem + L::kK + st * L::kKVBytes + dh * kSubTileBytes, &tm_k, &bars[BAR_K_FULL + st], dh * 64,
                      kvh, kv_begin + j * kBlockN);
        issued_k = j + 1;
        if (j >= 2) ok = mbar_wait(&bars[BAR_V_EMPTY + st], ((j >> 1) - 1) & 1, abort_flag);
        if (!ok) break;
        mbar_arrive_expect_tx(&bars[BAR_V_FULL + st], L::kKVBytes);
        for (int dh = 0; dh < L::kDSub; ++dh)
          tma_load_3d(smem + L::kV + st * L::kKVBytes + dh * kSubTileBytes, &tm_v, &bars[BAR_V_FULL + st], dh * 64,
                      kvh, kv_begin + j * kBlockN);
        issued_v = j + 1;
      }
      if (!ok) {
        // Let every copy that was issued land before shared memory is released.
        mbar_wait_drain(&bars[BAR_Q_FULL], 0);
        for (int j = max(0, issued_k - 2); j < issued_k; ++j) mbar_wait_drain(&bars[BAR_K_FULL + (j & 1)], (j >> 1) & 1);
        for (int j = max(0, issued_v - 2); j < issued_v; ++j) mbar_wait_drain(&bars[BAR_V_FULL + (j & 1)], (j >> 1) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ======================= MMA issuer =======================
    if (lane == 0 && nblk > 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(kBlockM, kBlockN, false, false);
      constexpr uint32_t idesc_o = idesc_bf16_f32(kBlockM, D, false, true);
      const uint32_t sQ = smem_u32(smem + L::kQ);
      const uint32_t sK = smem_u32(smem + L::kK);
      const uint32_t sV = smem_u32(smem + L::kV);
      const uint32_t sP = smem_u32(smem + L::kP);
      bool ok = mbar_wait(&bars[BAR_Q_FULL], 0, abort_flag);
      for (int j = 0; j <= nblk && ok; ++j) {
        if (j < nblk) {
          const int b = j & 1;
          ok = mbar_wait(&bars[BAR_K_FULL + b], (j >> 1) & 1, abort_flag);
          if (ok && j >= 2) ok = mbar_wait(&bars[BAR_S_FREE + b], ((j >> 1) - 1) & 1, abort_flag);
          if (!ok) break;
          tc_fence_after_sync();
          const uint32_t kbase = sK + b * L::kKVBytes;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kSubTileBytes + (kk & 3) * 32;
            umma_bf16_ss(tS0 + b * 128, sdesc_sw128(sQ + off, 16, 1024), sdesc_sw128(kbase + off, 16, 1024), idesc_s,
                         kk > 0);
          }
          umma_commit(&bars[BAR_S_FULL + b]);
          umma_commit(&bars[BAR_K_EMPTY + b]);
        }
        if (j >= 1) {
          const int jj = j - 1;
          const int b = jj & 1;
          ok = mbar_wait(&bars[BAR_P_FULL], jj & 1, abort_flag);
          if (ok) ok = mbar_wait(&bars[BAR_V_FULL + b], (jj >> 1) & 1, abort_flag);
          if (!ok) break;
          tc_fence_after_sync();
          const uint32_t vbase = sV + b * L::kKVBytes;
#pragma unroll
          for (int kk = 0; kk < kBlockN / 16; ++kk) {
            const uint32_t poff = (kk >> 2) * kSubTileBytes + (kk & 3) * 32;
            umma_bf16_ss(tO, sdesc_sw128(sP + poff, 16, 1024), sdesc_sw128(vbase + kk * 2048, kSubTileBytes, 1024),
                         idesc_o, (jj > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(&bars[BAR_O_READY]);
          umma_commit(&bars[BAR_V_EMPTY + b]);
        }
      }
      // All MMAs issued by this thread complete before TMEM can be released.
      umma_commit(&bars[BAR_DRAIN]);
      mbar_wait_drain(&bars[BAR_DRAIN], 0);
    }
    __syncwarp();
  } else {
    // ======================= softmax / correction / epilogue =======================
    const int r = threadIdx.x;  // query row == TMEM lane
    const int t_loc = r / G;
    const int g = r - t_loc * G;
    const bool row_valid = (r < rows_used) && (t_loc < n_tok_valid);
    const int qpos = q0_local + t_loc;  // prefill: position in the sequence
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t sP = smem_u32(smem + L::kP);
    float m_run = -INFINITY;  // running max, log2 domain (scaled)
    float l_run = 0.f;
    bool ok = true;

    for (int j = 0; j < nblk; ++j) {
      const int b = j & 1;
      ok = warp_wait(&bars[BAR_S_FULL + b], (j >> 1) & 1, abort_flag);
      if (!ok) break;
      tc_fence_after_sync();
      float s[kBlockN];
#pragma unroll
      for (int c = 0; c < kBlockN / 32; ++c) {
        uint32_t raw[32];
        tmem_ld32(tS0 + b * 128 + c * 32 + lane_off, raw);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(raw[i]);
      }
      tc_fence_before_sync();
      mbar_arrive(&bars[BAR_S_FREE + b]);

      // Masking: keys past the tile's reach (decode: past the prefix; prefill:
      // later than the query, which also covers keys past the sequence end).
      const int key0 = j * kBlockN;
      int lim;  // last valid key column in this block for this row
      if constexpr (MODE == AttnMode::kPrefill) lim = qpos - key0;
      else lim = p.Lp - 1 - key0;
      if (lim < kBlockN - 1) {
#pragma unroll
        for (int c = 0; c < kBlockN; ++c)
          if (c > lim) s[c] = -INFINITY;
      }
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < kBlockN; ++c) mx = fmaxf(mx, s[c]);
      const float m_cand = mx * p.scale_log2;
      float m_new = m_run;
      if (m_cand > m_run + kLazyRescaleLog2) m_new = m_cand;
      const float alpha = exp2_approx(m_run - m_new);  // 0 on the first block, 1 when unchanged
      const bool rescale_o = (j > 0) && (m_new != m_run);
      m_run = m_new;

      float lsum = 0.f;
      uint32_t pk[kBlockN / 2];
#pragma unroll
      for (int c = 0; c < kBlockN; c += 2) {
        const float p0 = exp2_approx(fmaf(s[c], p.scale_log2, -m_new));
        const float p1 = exp2_approx(fmaf(s[c + 1], p.scale_log2, -m_new));
        lsum += p0 + p1;
        pk[c >> 1] = pack_bf16x2(p0, p1);
      }
      l_run = l_run * alpha + lsum;

      // P's buffer and O are free once the previous block's P.V has completed.
      if (j > 0) {
        ok = warp_wait(&bars[BAR_O_READY], (j - 1) & 1, abort_flag);
        if (!ok) break;
        tc_fence_after_sync();
        if (__any_sync(0xffffffffu, rescale_o)) {
          const float a = rescale_o ? alpha : 1.f;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t raw[32];
            tmem_ld32(tO + c * 32 + lane_off, raw);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) raw[i] = __float_as_uint(__uint_as_float(raw[i]) * a);
            tmem_st32(tO + c * 32 + lane_off, raw);
          }
          tmem_wait_st();
        }
      }
      // P (bf16) -> shared memory, K-major 128-byte swizzle, 2 blocks of 64 keys.
#pragma unroll
      for (int ch = 0; ch < kBlockN / 8; ++ch) {
        const uint32_t addr = sP + (ch >> 3) * kSubTileBytes + r * 128 + ((((ch & 7) ^ (r & 7)) & 7) << 4);
        st_shared_v4(addr, pk[ch * 4 + 0], pk[ch * 4 + 1], pk[ch * 4 + 2], pk[ch * 4 + 3]);
      }
      fence_proxy_async_smem();
      tc_fence_before_sync();
      mbar_arrive(&bars[BAR_P_FULL]);
    }

    // ---- epilogue ----
    if (ok && nblk > 0) ok = warp_wait(&bars[BAR_O_READY], (nblk - 1) & 1, abort_flag);
    if (ok) {
      tc_fence_after_sync();
      float acc[D];
      if (nblk > 0) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t raw[32];
          tmem_ld32(tO + c * 32 + lane_off, raw);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) acc[c * 32 + i] = __uint_as_float(raw[i]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < D; ++i) acc[i] = 0.f;
      }

      if constexpr (MODE == AttnMode::kDecodePrefix) {
        // Suffix keys of this beam on CUDA cores: its parent's history rows
        // then its own new row, merged into the same online-softmax state.
        const int beam = row0_global + t_loc;
        // The Q tile is read below through the generic proxy: wait for its copy.
        ok = warp_wait(&bars[BAR_Q_FULL], 0, abort_flag);
        if (ok && row_valid) {
          int src = beam;
          if (p.parent) {
            src = p.parent[beam];
            if (src < 0 || src >= p.W) {
              if (p.dev_status) atomicOr(p.dev_status, kDevBadParent);
              src = 0;
            }
          }
          // q row from the swizzled Q tile in shared memory
          float q[D];
#pragma unroll
          for (int d = 0; d < D; d += 8) {
            const uint4 v = *reinterpret_cast<const uint4*>(smem + L::kQ + (d >> 6) * kSubTileBytes +
                                                             sw128_offset(r, d & 63));
            const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 f = __bfloat1622float2(h2[i]);
              q[d + 2 * i] = f.x;
              q[d + 2 * i + 1] = f.y;
            }
          }
          const int n_suffix = p.L_prev + (p.k_new != nullptr ? 1 : 0);
          const int64_t row_stride = static_cast<int64_t>(p.n_kv_heads) * D;
          for (int sidx = 0; sidx < n_suffix; ++sidx) {
            const __nv_bfloat16* krow;
            const __nv_bfloat16* vrow;
            if (sidx < p.L_prev) {
              krow = p.ks + (static_cast<int64_t>(src) * p.Smax + sidx) * row_stride + kvh * D;
              vrow = p.vs + (static_cast<int64_t>(src) * p.Smax + sidx) * row_stride + kvh * D;
            } else {
              krow = p.k_new + static_cast<int64_t>(beam) * row_stride + kvh * D;
              vrow = p.v_new + static_cast<int64_t>(beam) * row_stride + kvh * D;
            }
            float dot = 0.f;
#pragma unroll
            for (int d = 0; d < D; d += 8) {
              const uint4 kv = __ldg(reinterpret_cast<const uint4*>(krow + d));
              const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&kv);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float2 f = __bfloat1622float2(h2[i]);
                dot = fmaf(q[d + 2 * i], f.x, dot);
                dot = fmaf(q[d + 2 * i + 1], f.y, dot);
              }
            }
            const float sc = dot * p.scale_log2;
            const float m_new = fmaxf(m_run, sc);
            const float alpha = exp2_approx(m_run - m_new);
            const float pw = exp2_approx(sc - m_new);
            l_run = l_run * alpha + pw;
#pragma unroll
            for (int d = 0; d < D; d += 8) {
              const uint4 vv = __ldg(reinterpret_cast<const uint4*>(vrow + d));
              const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&vv);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float2 f = __bfloat1622float2(h2[i]);
                acc[d + 2 * i] = fmaf(acc[d + 2 * i], alpha, pw * f.x);
                acc[d + 2 * i + 1] = fmaf(acc[d + 2 * i + 1], alpha, pw * f.y);
              }
            }
            m_run = m_new;
          }
        }
      }

      if (ok && row_valid) {
        const float inv_l = 1.f / l_run;
        const int h = kvh * G + g;
        // index of (token or beam, q head) in O
        const int64_t out_row = static_cast<int64_t>(row0_global + t_loc) * p.n_q_heads + h;
        uint4* dst = reinterpret_cast<uint4*>(p.o + out_row * D);
#pragma unroll
        for (int d = 0; d < D; d += 8) {
          uint4 v;
          v.x = pack_bf16x2(acc[d + 0] * inv_l, acc[d + 1] * inv_l);
          v.y = pack_bf16x2(acc[d + 2] * inv_l, acc[d + 3] * inv_l);
          v.z = pack_bf16x2(acc[d + 4] * inv_l, acc[d + 5] * inv_l);
          v.w = pack_bf16x2(acc[d + 6] * inv_l, acc[d + 7] * inv_l);
          dst[d >> 3] = v;
        }
        if (p.lse) {
          const float lse = (m_run + __log2f(l_run)) * 0.69314718055994531f;
          if constexpr (MODE == AttnMode::kPrefill)
            p.lse[static_cast<int64_t>(h) * p.total_tokens + row0_global + t_loc] = lse;
          else
            p.lse[out_row] = lse;
        }
      }
    }

    if constexpr (MODE == AttnMode::kDecodePrefix) {
      // Suffix reorder for this tile's beams and KV head:
      //   out[b, s] = in[parent[b], s] (s < L_prev), out[b, L_prev] = new[b].
      const int n_suffix = p.L_prev + (p.k_new != nullptr ? 1 : 0);
      const int64_t row_stride = static_cast<int64_t>(p.n_kv_heads) * D;
      const int items = n_tok_valid * n_suffix * (D / 8);
      for (int it = threadIdx.x; it < items; it += 128) {
        const int chunk = it % (D / 8);
        const int rest = it / (D / 8);
        const int sidx = rest % n_suffix;
        const int beam = row0_global + rest / n_suffix;
        int src = p.parent ? p.parent[beam] : beam;
        if (src < 0 || src >= p.W) src = 0;  // flagged above
        const int64_t dst_off = (static_cast<int64_t>(beam) * p.Smax + sidx) * row_stride + kvh * D + chunk * 8;
        uint4 kv, vv;
        if (sidx < p.L_prev) {
          const int64_t src_off = (static_cast<int64_t>(src) * p.Smax + sidx) * row_stride + kvh * D + chunk * 8;
          kv = __ldg(reinterpret_cast<const uint4*>(p.ks + src_off));
          vv = __ldg(reinterpret_cast<const uint4*>(p.vs + src_off));
        } else {
          const int64_t src_off = static_cast<int64_t>(beam) * row_stride + kvh * D + chunk * 8;
          kv = __ldg(reinterpret_cast<const uint4*>(p.k_new + src_off));
          vv = __ldg(reinterpret_cast<const uint4*>(p.v_new + src_off));
        }
        *reinterpret_cast<uint4*>(p.ks_out + dst_off) = kv;
        *reinterpret_cast<uint4*>(p.vs_out + dst_off) = vv;
      }
    }
  }

  // ---- teardown ----
  tc_fence_before_sync();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag && p.dev_status) atomicOr(p.dev_status, kDevPipelineTimeout);
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace slm
