// Blackwell (sm_103a) attention core shared by packed prefill and the
// shared-prefix decode.
//
// A persistent CTA per SM walks a list of work units.  A unit is two query
// sub-tiles of 128 rows that read the same keys: rows are (token, head)
// pairs -- TOK = 128 / G consecutive tokens (prefill: positions of one
// sequence; decode: beams) times the G query heads that share one KV head, so
// each K/V block is loaded once for 2 x G heads ("Triton Packed GQA" in
// section 3.1 of the article "SLM 生成式高并发推理引擎：延迟约束下的有效吞吐优化" does not
// expand K/V heads either).
//
// Warp roles (320 threads):
//   warps 0-3  softmax of sub-tile 0 (thread = query row = TMEM lane)
//   warps 4-7  softmax of sub-tile 1
//   warp  8    TMA producer: lane 1 loads Q tiles (two buffers across units
//              at D = 64, one at D = 128), lane 0 a ring of K/V blocks,
//              128-byte swizzled
//   warp  9    tcgen05 issuer: S_t = Q_t K^T into TMEM, then O_t += P_t V
//              with P_t read back from TMEM where the softmax wrote it over
//              S_t (bf16, two per column)
//
// Per key block the issue order is PV_0(j), S_0(j+1), PV_1(j), S_1(j+1), so
// each sub-tile's softmax overlaps the other sub-tile's MMAs.  tcgen05 work
// completes in issue order, so a softmax that sees S_t(j+1) done also knows
// PV_t(j) is done and may rescale O_t.  The online softmax keeps its running
// maximum until a block raises it by more than 2^8 (the factor cancels in the
// final division), so O is rarely rescaled.
//
// The kernel runs as a programmatic dependent of the one before it (prefill:
// its schedule kernel): setup first, griddepcontrol.wait before any global
// memory is read.  Decode can
// split the prompt's key blocks over several CTAs per beam tile: each split
// leaves its rows' partial softmax state in a caller workspace and the last
// one to finish (atomic ticket) merges them before the suffix keys.
//
// Every mbarrier wait is bounded (see sm103_ptx.cuh); a stuck pipeline ends
// the kernel with a status bit instead of a hang.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "slm_internal.h"
#include "sm103_ptx.cuh"

namespace slm {

constexpr int kBlockM = 128;              // query rows per sub-tile (TMEM lanes)
constexpr int kBlockN = 128;              // keys per block
constexpr int kFwdThreads = 320;
constexpr int kSubTileBytes = 128 * 128;  // 128 rows x 64 bf16, one swizzle block column
constexpr uint32_t kTmemCols = 512;
constexpr float kLazyRescaleLog2 = 8.0f;

enum class AttnMode : int { kPrefill = 0, kDecodePrefix = 1 };

struct AttnParams {
  int n_q_heads, n_kv_heads, group, tok_per_tile;
  float scale_log2;          // softmax_scale * log2(e)
  __nv_bfloat16* o;
  float* o_f32;              // fp32 O rows (kernels instantiated with F32OUT only)
  float* lse;                // nullable
  int32_t* dev_status;       // nullable
  uint64_t wait_ns;          // limit of every bounded mbarrier wait
  // prefill: each softmax warp writes its 32 rows (32 / G whole tokens) with
  // TMA stores through a {64, G, 32 / G} box of tm_o (G divides 32)
  int warp_tma_store;
  // prefill
  const int32_t* cu_seqlens;
  const int32_t* items;      // [0] = count, then (start, length, pair) per item, longest sequences first
  int items_cap;             // items the workspace holds
  int total_tokens;
  // decode
  const __nv_bfloat16* q;    // read by the suffix merge
  const __nv_bfloat16* ks;
  const __nv_bfloat16* vs;
  const __nv_bfloat16* k_new;  // nullable (no append)
  const __nv_bfloat16* v_new;
  const int32_t* parent;     // nullable (identity)
  __nv_bfloat16* ks_out;
  __nv_bfloat16* vs_out;
  int W, Lp, L_prev, Smax;
  // decode with the prompt's key blocks split over CTAs: every split writes
  // its rows' (max, sum, unnormalised O); the last split of a tile to finish
  // merges them and runs the epilogue.  n_split = 1: no split.
  // Parts are stored per sub-tile and column, rows innermost, so that the
  // 128 threads of a sub-tile read and write them coalesced.
  int n_split, blk_per_split;
  float* ws_o;          // [n_split][tiles * n_kv_heads * 2][D][128]
  float2* ws_ml;        // [n_split][tiles * n_kv_heads * 2][128]
  int32_t* tickets;     // [tiles * n_kv_heads * 2][4 warps]: zero between calls
  int64_t ws_o_elems;   // floats in ws_o (bounds checks of debug builds)
  int tickets_cap;      // ints in tickets
};

// Decode (D = 64): each softmax warp stages its beams' suffix rows (the
// parents' history rows and the new rows, K and V, of its KV head) in its
// own 8 KB, loaded with cp.async as the unit starts, so the suffix merge in
// the epilogue reads shared memory instead of waiting on dependent loads.
constexpr int kHistWarpBytes = 8192;

template <int D, AttnMode MODE = AttnMode::kPrefill>
struct FwdSmem {
  static constexpr int kDSub = D / 64;
  static constexpr int kTile = kDSub * kSubTileBytes;  // 128 rows x D bf16
  // D = 128: one Q buffer, released as soon as the unit's last S MMA is done,
  // so the K/V ring can hold 2 blocks and the next unit's first blocks
  // arrive while the current unit ends.  D = 64: two Q buffers, 4 blocks
  // (prefill) or 2 blocks and the suffix staging (decode).  Both: 32 KB to
  // stage O for TMA stores.
  static constexpr bool kHistStage = (MODE == AttnMode::kDecodePrefix) && (D == 64);
  static constexpr int kQBufs = (D == 128) ? 1 : 2;
  static constexpr int kStages = (D == 128) ? 4 : (kHistStage ? 4 : 8);  // K/V ring
  static constexpr int kQ = 0;                         // [kQBufs buffers][2 sub-tiles]
  static constexpr int kKV = kQ + 2 * kQBufs * kTile;
  static constexpr int kOut = kKV + kStages * kTile;   // [2 sub-tiles] 128 rows x 64 bf16: O staging for TMA stores
  static constexpr int kHist = kOut + 2 * kSubTileBytes;  // [8 softmax warps] suffix rows (decode, D = 64)
  static constexpr int kBar = kHist + (kHistStage ? 8 * kHistWarpBytes : 0);
  // barrier slots
  static constexpr int Q_FULL = 0, Q_EMPTY = 2, KV_FULL = 4, KV_EMPTY = KV_FULL + kStages,
                       S_FULL = KV_EMPTY + kStages, P_FULL = S_FULL + 2, O_FULL = P_FULL + 2,
                       O_EMPTY = O_FULL + 2, DRAIN = O_EMPTY + 2, kNumBars = DRAIN + 1;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kTotal = kMisc + 64;
  static constexpr int kAlloc = kTotal + 1024;  // room to align the base to 1024 bytes
};

struct UnitInfo {
  int kvh;
  int kv_begin;   // first key row (global index into K/V)
  int row0[2];    // first token (prefill) or beam (decode) of each sub-tile
  int q0[2];      // prefill: position of the sub-tile's first token in its sequence
  int n_tok[2];   // valid tokens / beams of each sub-tile
  int nblk[2];    // key blocks each sub-tile reads
  int nblk_max;
  int tile, split;  // decode: beam tile pair and key split of the unit
};

template <AttnMode MODE>
__device__ __forceinline__ int num_units(const AttnParams& p) {
  if constexpr (MODE == AttnMode::kPrefill) {
    const int n = p.items[0];
    return (in_bounds(n >= 0 && n <= p.items_cap, p.dev_status) ? n : 0) * p.n_kv_heads;
  }
  else return ((p.W + 2 * p.tok_per_tile - 1) / (2 * p.tok_per_tile)) * p.n_kv_heads * p.n_split;
}

// The memory part of a unit's description: the (start, length, pair) item
// of prefill.  Loaded a whole unit ahead and only combined when needed, so
// the load latency hides behind the current unit.
struct UnitRaw {
  int s0, len, pair;
};

template <AttnMode MODE>
__device__ __forceinline__ UnitRaw unit_raw(const AttnParams& p, int u) {
  UnitRaw r{0, 0, 0};
  if constexpr (MODE == AttnMode::kPrefill) {
    const int item = u / p.n_kv_heads;
    r.s0 = __ldg(&p.items[1 + 3 * item]);
    r.len = __ldg(&p.items[2 + 3 * item]);
    r.pair = __ldg(&p.items[3 + 3 * item]);
  }
  return r;
}

template <AttnMode MODE>
__device__ __forceinline__ UnitInfo unit_info(const AttnParams& p, int u, const UnitRaw& raw) {
  UnitInfo U;
  const int TOK = p.tok_per_tile;
  U.kvh = u % p.n_kv_heads;
  const int item = u / p.n_kv_heads;
  if constexpr (MODE == AttnMode::kPrefill) {
    const int s0 = raw.s0;
    const int len = raw.len;
    const int pair = raw.pair;
    U.kv_begin = s0;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      U.q0[t] = (2 * pair + t) * TOK;
      U.n_tok[t] = max(0, min(TOK, len - U.q0[t]));
      U.row0[t] = s0 + U.q0[t];
      U.nblk[t] = U.n_tok[t] > 0 ? (U.q0[t] + U.n_tok[t] + kBlockN - 1) / kBlockN : 0;
    }
    U.tile = item;
    U.split = 0;
    // a work item must lie inside its sequence and the sequence inside the batch
    if (!in_bounds(s0 >= 0 && len >= 1 && s0 + len <= p.total_tokens && pair >= 0 && 2 * pair * TOK < len,
                   p.dev_status)) {
#pragma unroll
      for (int t = 0; t < 2; ++t) U.n_tok[t] = U.nblk[t] = 0;
    }
  } else {
    U.split = item % p.n_split;
    U.tile = item / p.n_split;
    const int b0 = U.split * p.blk_per_split;
    const int nb = max(0, min(p.blk_per_split, (p.Lp + kBlockN - 1) / kBlockN - b0));
    U.kv_begin = b0 * kBlockN;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      U.q0[t] = 0;
      U.row0[t] = (2 * U.tile + t) * TOK;
      U.n_tok[t] = max(0, min(TOK, p.W - U.row0[t]));
      U.nblk[t] = U.n_tok[t] > 0 ? nb : 0;
    }
  }
  U.nblk_max = max(U.nblk[0], U.nblk[1]);
  return U;
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          uint64_t limit_ns) {
  bool ok = mbar_wait(bar, parity, abort_flag, limit_ns);
  return __all_sync(0xffffffffu, ok);
}

// F32OUT: O is written as fp32 rows to p.o_f32 (the test and diagnostic
// entry points) instead of bf16; a separate instantiation, so that the fp32
// store path costs the bf16 kernels no registers.
template <int D, AttnMode MODE, bool F32OUT = false>
__global__ void __launch_bounds__(kFwdThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    const AttnParams p) {
  using L = FwdSmem<D, MODE>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t wlim = p.wait_ns;
  const int G = p.group;
  const int TOK = p.tok_per_tile;
  const int rows_used = TOK * G;
  // decode: the units are known from the arguments; CTAs beyond them leave
  const int n_units_dec = (MODE == AttnMode::kPrefill) ? 0 : num_units<MODE>(p);
  if (MODE != AttnMode::kPrefill && static_cast<int>(blockIdx.x) >= n_units_dec) return;

  auto q_tile = [&](int qb, int t) { return smem + L::kQ + (qb * 2 + t) * L::kTile; };
  auto kv_tile = [&](uint32_t slot) { return smem + L::kKV + slot * L::kTile; };

  // ---- setup ---------------------------------------------------------------
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[L::Q_FULL + i], 1);
      mbar_init(&bars[L::Q_EMPTY + i], 1);
      mbar_init(&bars[L::S_FULL + i], 1);
      mbar_init(&bars[L::P_FULL + i], 128);
      mbar_init(&bars[L::O_FULL + i], 1);
      mbar_init(&bars[L::O_EMPTY + i], 128);
    }
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(&bars[L::KV_FULL + s], 1);
      mbar_init(&bars[L::KV_EMPTY + s], 1);
    }
    mbar_init(&bars[L::DRAIN], 1);
    fence_mbarrier_init();
  }
  if (warp == 8 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    if (MODE == AttnMode::kPrefill) tma_prefetch_desc(&tm_o);
    if (MODE == AttnMode::kPrefill || p.Lp > 0) {  // the K/V maps are left empty when there is no prefix
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
    }
  }
  // Rows of the Q tiles the TMA box never covers (G not dividing 128) must
  // hold finite values: zero them once.
  if (rows_used < kBlockM) {
    const int tail = kBlockM - rows_used;
    for (int i = threadIdx.x; i < 2 * L::kQBufs * L::kDSub * tail * 8; i += kFwdThreads) {
      const int chunk = i & 7;
      int rest = i >> 3;
      const int r = rows_used + rest % tail;
      rest /= tail;
      const int sub = rest % L::kDSub;
      const int tile = rest / L::kDSub;
      *reinterpret_cast<uint4*>(smem + L::kQ + tile * L::kTile + sub * kSubTileBytes + r * 128 + chunk * 16) =
          make_uint4(0, 0, 0, 0);
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
  // A programmatic dependent of the kernel before it (prefill: its schedule
  // kernel): the setup above overlaps that kernel, global memory is read only
  // after this.  A CTA beyond the last unit runs empty loops and frees its
  // TMEM.
  pdl_wait();
  pdl_launch_dependents();
  const int n_units = (MODE == AttnMode::kPrefill) ? num_units<MODE>(p) : n_units_dec;

  if (warp == 8) {
    // ======================= TMA producer =======================
    // Two lanes, each blocking only on its own resource (independent thread
    // scheduling lets them progress separately): lane 1 streams the Q tiles
    // into the two Q buffers, as far ahead as the buffers allow; lane 0
    // streams K/V blocks through the ring.
    if (lane == 1) {
      int qi = 0;
      bool ok = true;
      UnitRaw rn = unit_raw<MODE>(p, blockIdx.x);
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        const UnitInfo U = unit_info<MODE>(p, u, rn);
        if (u + static_cast<int>(gridDim.x) < n_units) rn = unit_raw<MODE>(p, u + gridDim.x);
        if (U.nblk_max == 0) continue;  // decode with an empty prefix: suffix only
        const int qb = qi % L::kQBufs;
        if (qi >= L::kQBufs) ok = mbar_wait(&bars[L::Q_EMPTY + qb], ((qi / L::kQBufs) - 1) & 1, abort_flag, wlim);
        if (!ok) break;
        uint32_t q_bytes = 0;
        for (int t = 0; t < 2; ++t)
          if (U.n_tok[t] > 0) q_bytes += static_cast<uint32_t>(L::kDSub) * 64u * G * TOK * 2u;
        mbar_arrive_expect_tx(&bars[L::Q_FULL + qb], q_bytes);
        for (int t = 0; t < 2; ++t)
          if (U.n_tok[t] > 0)
            for (int dh = 0; dh < L::kDSub; ++dh)
              tma_load_3d(q_tile(qb, t) + dh * kSubTileBytes, &tm_q, &bars[L::Q_FULL + qb], dh * 64, U.kvh * G,
                          U.row0[t]);
        ++qi;
      }
      if (!ok)  // let the copies already issued land before shared memory is released
        for (int i = qi > L::kQBufs ? qi - L::kQBufs : 0; i < qi; ++i)
          mbar_wait_drain(&bars[L::Q_FULL + (i % L::kQBufs)], (i / L::kQBufs) & 1);
    } else if (lane == 0) {
      uint32_t kv_i = 0;
      bool ok = true;
      UnitRaw rn = unit_raw<MODE>(p, blockIdx.x);
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        const UnitInfo U = unit_info<MODE>(p, u, rn);
        if (u + static_cast<int>(gridDim.x) < n_units) rn = unit_raw<MODE>(p, u + gridDim.x);
        for (int j = 0; j < U.nblk_max && ok; ++j) {
          for (int kind = 0; kind < 2; ++kind) {
            const uint32_t slot = kv_i % L::kStages, use = kv_i / L::kStages;
            if (use >= 1) ok = mbar_wait(&bars[L::KV_EMPTY + slot], (use - 1) & 1, abort_flag, wlim);
            if (!ok) break;
            mbar_arrive_expect_tx(&bars[L::KV_FULL + slot], L::kTile);
            for (int dh = 0; dh < L::kDSub; ++dh)
              tma_load_3d(kv_tile(slot) + dh * kSubTileBytes, kind ? &tm_v : &tm_k, &bars[L::KV_FULL + slot],
                          dh * 64, U.kvh, U.kv_begin + j * kBlockN);
            ++kv_i;
          }
        }
      }
      if (!ok)
        for (uint32_t i = kv_i > static_cast<uint32_t>(L::kStages) ? kv_i - L::kStages : 0; i < kv_i; ++i)
          mbar_wait_drain(&bars[L::KV_FULL + i % L::kStages], (i / L::kStages) & 1);
    }
    __syncwarp();
  } else if (warp == 9) {
    // ======================= tcgen05 issuer =======================
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(kBlockM, kBlockN, false, false);
      constexpr uint32_t idesc_o = idesc_bf16_f32(kBlockM, D, false, true);
      uint32_t kv_i = 0, p_cnt[2] = {0, 0}, o_used[2] = {0, 0};
      int it = 0;
      bool ok = true;
      auto slot = [&](uint32_t i) { return i % L::kStages; };
      auto phase = [&](uint32_t i) { return (i / L::kStages) & 1; };
      auto issue_s = [&](int qb, int t, uint32_t kslot) {
        const uint32_t qa = smem_u32(q_tile(qb, t)), ka = smem_u32(kv_tile(kslot));
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kSubTileBytes + (kk & 3) * 32;
          umma_bf16_ss(tmem_base + t * 128, sdesc_sw128(qa + off, 16, 1024), sdesc_sw128(ka + off, 16, 1024),
                       idesc_s, kk > 0);
        }
      };
      auto issue_pv = [&](int t, uint32_t vslot, bool accumulate) {
        const uint32_t va = smem_u32(kv_tile(vslot));
#pragma unroll
        for (int kk = 0; kk < kBlockN / 16; ++kk)
          umma_bf16_ts(tmem_base + 256 + t * 128, tmem_base + t * 128 + kk * 8,
                       sdesc_sw128(va + kk * 2048, kSubTileBytes, 1024), idesc_o, (accumulate || kk > 0) ? 1u : 0u);
      };
      UnitRaw rn = unit_raw<MODE>(p, blockIdx.x);
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        const UnitInfo U = unit_info<MODE>(p, u, rn);
        // the next unit's item loads while this one runs
        if (u + static_cast<int>(gridDim.x) < n_units) rn = unit_raw<MODE>(p, u + gridDim.x);
        if (U.nblk_max == 0) continue;
        const int qb = it % L::kQBufs;
        ok = mbar_wait(&bars[L::Q_FULL + qb], (it / L::kQBufs) & 1, abort_flag, wlim);
        const uint32_t kbase = kv_i;
        if (ok) ok = mbar_wait(&bars[L::KV_FULL + slot(kbase)], phase(kbase), abort_flag, wlim);
        if (!ok) break;
        tc_fence_after_sync();
        for (int t = 0; t < 2; ++t)
          if (U.nblk[t] > 0) {
            issue_s(qb, t, slot(kbase));
            umma_commit(&bars[L::S_FULL + t]);
          }
        umma_commit(&bars[L::KV_EMPTY + slot(kbase)]);
        if (U.nblk_max == 1) umma_commit(&bars[L::Q_EMPTY + qb]);  // the unit's last S MMAs are issued
        for (int j = 0; j < U.nblk_max && ok; ++j) {
          const uint32_t vi = kbase + 2 * j + 1, kn = kbase + 2 * j + 2;
          ok = mbar_wait(&bars[L::KV_FULL + slot(vi)], phase(vi), abort_flag, wlim);
          bool k_next_ready = false;  // K_{j+1} is waited for only by the S that needs it
          for (int t = 0; t < 2 && ok; ++t) {
            if (j >= U.nblk[t]) continue;
            if (j == 0 && o_used[t] > 0) ok = mbar_wait(&bars[L::O_EMPTY + t], (o_used[t] - 1) & 1, abort_flag, wlim);
            if (ok) ok = mbar_wait(&bars[L::P_FULL + t], p_cnt[t] & 1, abort_flag, wlim);
            if (!ok) break;
            ++p_cnt[t];
            tc_fence_after_sync();
            issue_pv(t, slot(vi), j > 0);
            if (j == U.nblk[t] - 1) {
              umma_commit(&bars[L::O_FULL + t]);
              ++o_used[t];
            } else {
              if (!k_next_ready) {
                ok = mbar_wait(&bars[L::KV_FULL + slot(kn)], phase(kn), abort_flag, wlim);
                if (!ok) break;
                tc_fence_after_sync();
                k_next_ready = true;
              }
              issue_s(qb, t, slot(kn));
              umma_commit(&bars[L::S_FULL + t]);
            }
          }
          if (!ok) break;
          umma_commit(&bars[L::KV_EMPTY + slot(vi)]);
          if (j + 1 < U.nblk_max) umma_commit(&bars[L::KV_EMPTY + slot(kn)]);
          // the Q buffer is free once the unit's last S MMAs complete
          if (j + 1 == U.nblk_max - 1) umma_commit(&bars[L::Q_EMPTY + qb]);
        }
        kv_i = kbase + 2 * U.nblk_max;
        ++it;
      }
      // All MMAs issued by this thread complete before TMEM can be released.
      umma_commit(&bars[L::DRAIN]);
      mbar_wait_drain(&bars[L::DRAIN], 0);
    }
    __syncwarp();
  } else {
    // ======================= softmax / epilogue (two warpgroups) =======================
    const int t = warp >> 2;              // sub-tile of this warpgroup
    const int wq = warp & 3;              // rows 32 wq .. 32 wq + 31 of the sub-tile
    const int r = threadIdx.x & 127;      // query row == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem_base + t * 128;
    const uint32_t tO = tmem_base + 256 + t * 128;
    const int t_loc = r / G;
    const int g = r - t_loc * G;
    uint32_t s_cnt = 0, o_cnt = 0;
    bool ok = true;
    UnitRaw rn = unit_raw<MODE>(p, blockIdx.x);
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      const UnitInfo U = unit_info<MODE>(p, u, rn);
      if (u + static_cast<int>(gridDim.x) < n_units) rn = unit_raw<MODE>(p, u + gridDim.x);
      if (U.n_tok[t] == 0) continue;
      const bool row_valid = (r < rows_used) && (t_loc < U.n_tok[t]);
      const int qpos = U.q0[t] + t_loc;
      // Decode: this warp's beams' suffix rows, staged for the epilogue while
      // the prompt's blocks run (rows hb_first .. of the sub-tile; layout
      // [beam][suffix row][K, V][D]).
      bool hist_staged = false;
      int hb_first = 0;
      const uint8_t* hist_w = nullptr;
      if constexpr (L::kHistStage) {
        const int n_suffix = p.L_prev + (p.k_new != nullptr ? 1 : 0);
        hb_first = (32 * wq) / G;
        const int nb = min((32 * wq + 31) / G, U.n_tok[t] - 1) - hb_first + 1;
        hist_w = smem + L::kHist + (t * 4 + wq) * kHistWarpBytes;
        if (n_suffix > 0 && nb > 0 && nb <= 8 && nb * n_suffix * 2 * D * 2 <= kHistWarpBytes) {
          hist_staged = true;
          cp_async_wait_all();  // the last unit's copies into this region have landed
          int par = 0;          // parent of beam hb_first + lane
          if (lane < nb) {
            const int beam = U.row0[t] + hb_first + lane;
            par = p.parent ? __ldg(p.parent + beam) : beam;
            if (par < 0 || par >= p.W) par = 0;  // flagged by the epilogue
          }
          int pars[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) pars[k] = __shfl_sync(0xffffffffu, par, k);
          const int64_t row_stride = static_cast<int64_t>(p.n_kv_heads) * D;
          const int n_chunks = nb * n_suffix * 2 * (D / 8);
          for (int i = lane; i < n_chunks; i += 32) {
            const int c = i % (D / 8);
            const int rest = i / (D / 8);
            const int kind = rest & 1;
            const int sidx = (rest >> 1) % n_suffix;
            const int bb = (rest >> 1) / n_suffix;
            int sp = pars[0];
#pragma unroll
            for (int k = 1; k < 8; ++k)
              if (bb == k) sp = pars[k];
            const __nv_bfloat16* src;
            if (sidx < p.L_prev)
              src = (kind ? p.vs : p.ks) + (static_cast<int64_t>(sp) * p.Smax + sidx) * row_stride + U.kvh * D + c * 8;
            else
              src = (kind ? p.v_new : p.k_new) + static_cast<int64_t>(U.row0[t] + hb_first + bb) * row_stride +
                    U.kvh * D + c * 8;
            cp_async_16(const_cast<uint8_t*>(hist_w) + i * 16, src);
          }
          cp_async_commit();
        }
      }
      float m_run = -INFINITY;  // running max, log2 domain (scaled)
      float l_run = 0.f;
      for (int j = 0; j < U.nblk[t]; ++j) {
        ok = warp_wait(&bars[L::S_FULL + t], s_cnt & 1, abort_flag, wlim);
        if (!ok) break;
        ++s_cnt;
        tc_fence_after_sync();
        float s[kBlockN];
        {
          uint32_t raw[kBlockN];
#pragma unroll
          for (int c = 0; c < kBlockN / 32; ++c)
            tmem_ld32(tS + c * 32 + lane_off, *reinterpret_cast<uint32_t(*)[32]>(&raw[c * 32]));
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < kBlockN; ++i) s[i] = __uint_as_float(raw[i]);
        }
        // keys past the row's reach: later than the query (prefill; this
        // also covers keys past the sequence) or past the prefix (decode)
        const int key0 = j * kBlockN;
        int lim;
        if constexpr (MODE == AttnMode::kPrefill) lim = qpos - key0;
        else lim = p.Lp - 1 - (U.kv_begin + key0);
        if (lim < kBlockN - 1) {
#pragma unroll
          for (int c = 0; c < kBlockN; ++c)
            if (c > lim) s[c] = -INFINITY;
        }
        float mx8[8];  // eight independent max chains
#pragma unroll
        for (int i = 0; i < 8; ++i) mx8[i] = s[i];
#pragma unroll
        for (int c = 8; c < kBlockN; ++c) mx8[c & 7] = fmaxf(mx8[c & 7], s[c]);
        const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                               fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
        const float m_cand = mx * p.scale_log2;
        float m_new = m_run;
        if (m_cand > m_run + kLazyRescaleLog2) m_new = m_cand;
        const float alpha = exp2_approx(m_run - m_new);  // 0 on the first block, 1 when unchanged
        const bool rescale_o = (j > 0) && (m_new != m_run);
        m_run = m_new;
        float ls4[4] = {0.f, 0.f, 0.f, 0.f};  // four independent sum chains
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t pk[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float p0 = exp2_approx(fmaf(s[h * 64 + 2 * i], p.scale_log2, -m_new));
            const float p1 = exp2_approx(fmaf(s[h * 64 + 2 * i + 1], p.scale_log2, -m_new));
            ls4[i & 3] += p0 + p1;
            pk[i] = pack_bf16x2(p0, p1);
          }
          tmem_st32(tS + h * 32 + lane_off, pk);  // P over the first half of S's columns
        }
        l_run = l_run * alpha + ((ls4[0] + ls4[1]) + (ls4[2] + ls4[3]));
        // PV_t(j-1) completed before S_t(j) did, and PV_t(j) waits for P_FULL:
        // O_t is stable here.
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
        }
        tmem_wait_st();
        tc_fence_before_sync();
        mbar_arrive(&bars[L::P_FULL + t]);
      }
      if (!ok) break;

      // ---- epilogue ----
      float acc[D];
      if (U.nblk[t] > 0) {
        ok = warp_wait(&bars[L::O_FULL + t], o_cnt & 1, abort_flag, wlim);
        if (!ok) break;
        ++o_cnt;
        tc_fence_after_sync();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t raw[32];
          tmem_ld32(tO + c * 32 + lane_off, raw);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) acc[c * 32 + i] = __uint_as_float(raw[i]);
        }
        tc_fence_before_sync();
        mbar_arrive(&bars[L::O_EMPTY + t]);  // O_t may now take the next unit's products
      } else {
#pragma unroll
        for (int i = 0; i < D; ++i) acc[i] = 0.f;
      }
      const int h = U.kvh * G + g;
      const int rowid = U.row0[t] + t_loc;  // token (prefill) or beam (decode)

      if constexpr (MODE == AttnMode::kDecodePrefix) {
        if (p.n_split > 1) {
          // This split's part of each row goes to the workspace; for each warp's
          // 32 rows, the last split to arrive (ticket) merges all parts and goes
          // on, the others are done.  The last one also sets the ticket back to
          // zero.  Warps decide on their own: no barrier spans the warpgroup.
          const int64_t n_tt = static_cast<int64_t>((p.W + 2 * TOK - 1) / (2 * TOK)) * p.n_kv_heads * 2;
          const int tt = (U.tile * p.n_kv_heads + U.kvh) * 2 + t;
          if (!in_bounds((U.split * n_tt + tt + 1) * D * 128 <= p.ws_o_elems && tt * 4 + wq < p.tickets_cap,
                         p.dev_status))
            continue;
          {
            float* dst = p.ws_o + (U.split * n_tt + tt) * D * 128 + r;
#pragma unroll
            for (int d = 0; d < D; ++d) __stcg(dst + d * 128, acc[d]);
            __stcg(&p.ws_ml[(U.split * n_tt + tt) * 128 + r], make_float2(m_run, l_run));
          }
          __threadfence();
          __syncwarp();
          int last = 0;
          if (lane == 0) {
            int32_t* ticket = &p.tickets[tt * 4 + wq];
            last = atomicAdd(ticket, 1) == p.n_split - 1;
            if (last) *ticket = 0;  // no other split touches it in this call
          }
          if (!__shfl_sync(0xffffffffu, last, 0)) continue;
          __threadfence();
          if (row_valid) {
            float m = m_run;
            for (int s = 0; s < p.n_split; ++s)
              if (s != U.split) m = fmaxf(m, __ldcg(&p.ws_ml[(s * n_tt + tt) * 128 + r]).x);
            const float a = exp2_approx(m_run - m);
            l_run *= a;
#pragma unroll
            for (int d = 0; d < D; ++d) acc[d] *= a;
            for (int s = 0; s < p.n_split; ++s) {
              if (s == U.split) continue;
              const float2 ml = __ldcg(&p.ws_ml[(s * n_tt + tt) * 128 + r]);
              const float f = exp2_approx(ml.x - m);
              l_run = fmaf(ml.y, f, l_run);
              const float* src = p.ws_o + (s * n_tt + tt) * D * 128 + r;
#pragma unroll
              for (int d = 0; d < D; ++d) acc[d] = fmaf(__ldcg(src + d * 128), f, acc[d]);
            }
            m_run = m;
          }
        }
        // Suffix keys of this beam on CUDA cores: its parent's history rows
        // then its own new row, merged into the same online-softmax state.
        if (hist_staged) {
          cp_async_wait_all();
          __syncwarp();  // every lane's staged rows are visible to the warp
        }
        // A CTA with a single unit still holds its Q tile (buffer 0, never
        // reloaded): the q rows come from there instead of global memory.
        const bool q_in_smem = n_units <= static_cast<int>(gridDim.x) && U.nblk_max > 0;
        if (q_in_smem) {
          ok = warp_wait(&bars[L::Q_FULL], 0, abort_flag, wlim);  // completed long ago: orders the TMA's writes
          if (!ok) break;
        }
        if (row_valid) {
          int src = rowid;
          if (p.parent) {
            src = p.parent[rowid];
            if (src < 0 || src >= p.W) {
              if (p.dev_status) atomicOr(p.dev_status, kDevBadParent);
              src = 0;
            }
          }
          uint32_t q2[D / 2];  // the q row, packed bf16 pairs
          const __nv_bfloat16* qrow = p.q + (static_cast<int64_t>(rowid) * p.n_q_heads + h) * D;
#pragma unroll
          for (int d = 0; d < D; d += 8) {
            const uint4 v = q_in_smem ? ld_shared_v4(q_tile(0, t) + (d / 64) * kSubTileBytes + sw128_offset(r, d % 64))
                                      : __ldg(reinterpret_cast<const uint4*>(qrow + d));
            q2[d / 2 + 0] = v.x;
            q2[d / 2 + 1] = v.y;
            q2[d / 2 + 2] = v.z;
            q2[d / 2 + 3] = v.w;
          }
          const int n_suffix = p.L_prev + (p.k_new != nullptr ? 1 : 0);
          const int64_t row_stride = static_cast<int64_t>(p.n_kv_heads) * D;
          for (int sidx = 0; sidx < n_suffix; ++sidx) {
            const __nv_bfloat16* krow;
            const __nv_bfloat16* vrow;
            if (hist_staged) {
              krow = reinterpret_cast<const __nv_bfloat16*>(hist_w) + ((t_loc - hb_first) * n_suffix + sidx) * 2 * D;
              vrow = krow + D;
            } else if (sidx < p.L_prev) {
              krow = p.ks + (static_cast<int64_t>(src) * p.Smax + sidx) * row_stride + U.kvh * D;
              vrow = p.vs + (static_cast<int64_t>(src) * p.Smax + sidx) * row_stride + U.kvh * D;
            } else {
              krow = p.k_new + static_cast<int64_t>(rowid) * row_stride + U.kvh * D;
              vrow = p.v_new + static_cast<int64_t>(rowid) * row_stride + U.kvh * D;
            }
            float dot = 0.f;
#pragma unroll
            for (int d = 0; d < D; d += 8) {
              const uint4 kv = hist_staged ? ld_shared_v4(krow + d) : __ldg(reinterpret_cast<const uint4*>(krow + d));
              const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&kv);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float2 f = __bfloat1622float2(h2[i]);
                const float2 qf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&q2[d / 2 + i]));
                dot = fmaf(qf.x, f.x, dot);
                dot = fmaf(qf.y, f.y, dot);
              }
            }
            const float sc = dot * p.scale_log2;
            const float m_new = fmaxf(m_run, sc);
            const float alpha = exp2_approx(m_run - m_new);
            const float pw = exp2_approx(sc - m_new);
            l_run = l_run * alpha + pw;
#pragma unroll
            for (int d = 0; d < D; d += 8) {
              const uint4 vv = hist_staged ? ld_shared_v4(vrow + d) : __ldg(reinterpret_cast<const uint4*>(vrow + d));
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

      // Prefill: a warp whose 32 rows are whole tokens of the sequence writes
      // them by TMA stores -- staged in shared memory in the swizzled box
      // layout (row r = token * G + head, as the Q tile), 64 columns at a
      // time, whole lines instead of 16-byte pieces of 256-byte rows.  Each
      // warp has its own quarter of the sub-tile's staging buffer, so no
      // barrier spans the warpgroup.  Other rows are stored row by row.
      const int wtok = p.warp_tma_store ? 32 / G : 0;
      const bool tma_out = (MODE == AttnMode::kPrefill) && !F32OUT && p.warp_tma_store &&
                           (wq + 1) * wtok <= U.n_tok[t] &&
                           in_bounds(U.row0[t] + (wq + 1) * wtok <= p.total_tokens, p.dev_status);
      if (tma_out) {
        const float inv_l = (l_run > 0.f) ? 1.f / l_run : 0.f;
        uint8_t* stage = smem + L::kOut + t * kSubTileBytes;
#pragma unroll
        for (int dh = 0; dh < L::kDSub; ++dh) {
          if (lane == 0) bulk_wait_read0();  // this warp's previous store has read its rows
          __syncwarp();
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const int d = dh * 64 + c * 8;
            st_shared_v4(smem_u32(stage + sw128_offset(r, c * 8)), pack_bf16x2(acc[d + 0] * inv_l, acc[d + 1] * inv_l),
                         pack_bf16x2(acc[d + 2] * inv_l, acc[d + 3] * inv_l),
                         pack_bf16x2(acc[d + 4] * inv_l, acc[d + 5] * inv_l),
                         pack_bf16x2(acc[d + 6] * inv_l, acc[d + 7] * inv_l));
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(&tm_o, stage + wq * 32 * 128, dh * 64, U.kvh * G, U.row0[t] + wq * wtok);
            bulk_commit();
          }
        }
      }
      const int rows_total = (MODE == AttnMode::kPrefill) ? p.total_tokens : p.W;
      if (row_valid && in_bounds(rowid >= 0 && rowid < rows_total && h < p.n_q_heads, p.dev_status)) {
        const float inv_l = 1.f / l_run;
        const int64_t out_row = static_cast<int64_t>(rowid) * p.n_q_heads + h;
        if constexpr (F32OUT) {
          float4* dst = reinterpret_cast<float4*>(p.o_f32 + out_row * D);
#pragma unroll
          for (int d = 0; d < D; d += 4)
            dst[d >> 2] = make_float4(acc[d] * inv_l, acc[d + 1] * inv_l, acc[d + 2] * inv_l, acc[d + 3] * inv_l);
        } else if (!tma_out) {
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
        }
        if (p.lse) {
          const float lse = (m_run + __log2f(l_run)) * 0.69314718055994531f;
          if constexpr (MODE == AttnMode::kPrefill) p.lse[static_cast<int64_t>(h) * p.total_tokens + rowid] = lse;
          else p.lse[out_row] = lse;
        }
      }

      if constexpr (MODE == AttnMode::kDecodePrefix) {
        // Suffix reorder for this sub-tile's beams and KV head:
        //   out[b, s] = in[parent[b], s] (s < L_prev), out[b, L_prev] = new[b].
        // Each warp copies the beams whose first row it holds (the warp that
        // took the last split's ticket, when the prompt is split), from its
        // staged rows when it has them.
        const int n_suffix = p.L_prev + (p.k_new != nullptr ? 1 : 0);
        const int64_t row_stride = static_cast<int64_t>(p.n_kv_heads) * D;
        const int b_lo = min((32 * wq + G - 1) / G, U.n_tok[t]);
        const int b_hi = min((32 * (wq + 1) + G - 1) / G, U.n_tok[t]);
        if (hist_staged) {
          const int items = (b_hi - b_lo) * n_suffix * 2 * (D / 8);
          for (int i = lane; i < items; i += 32) {
            const int chunk = i % (D / 8);
            const int rest = i / (D / 8);
            const int kind = rest & 1;
            const int sidx = (rest >> 1) % n_suffix;
            const int bb = b_lo + (rest >> 1) / n_suffix;
            const uint4 v = ld_shared_v4(hist_w + ((((bb - hb_first) * n_suffix + sidx) * 2 + kind) * (D / 8) + chunk) * 16);
            const int64_t dst_off =
                (static_cast<int64_t>(U.row0[t] + bb) * p.Smax + sidx) * row_stride + U.kvh * D + chunk * 8;
            *reinterpret_cast<uint4*>((kind ? p.vs_out : p.ks_out) + dst_off) = v;
          }
        } else {
          const int items = (b_hi - b_lo) * n_suffix * (D / 8);
          for (int i = lane; i < items; i += 32) {
            const int chunk = i % (D / 8);
            const int rest = i / (D / 8);
            const int sidx = rest % n_suffix;
            const int beam = U.row0[t] + b_lo + rest / n_suffix;
            int src = p.parent ? p.parent[beam] : beam;
            if (src < 0 || src >= p.W) src = 0;  // flagged above
            const int64_t dst_off = (static_cast<int64_t>(beam) * p.Smax + sidx) * row_stride + U.kvh * D + chunk * 8;
            uint4 kv, vv;
            if (sidx < p.L_prev) {
              const int64_t src_off = (static_cast<int64_t>(src) * p.Smax + sidx) * row_stride + U.kvh * D + chunk * 8;
              kv = __ldg(reinterpret_cast<const uint4*>(p.ks + src_off));
              vv = __ldg(reinterpret_cast<const uint4*>(p.vs + src_off));
            } else {
              const int64_t src_off = static_cast<int64_t>(beam) * row_stride + U.kvh * D + chunk * 8;
              kv = __ldg(reinterpret_cast<const uint4*>(p.k_new + src_off));
              vv = __ldg(reinterpret_cast<const uint4*>(p.v_new + src_off));
            }
            *reinterpret_cast<uint4*>(p.ks_out + dst_off) = kv;
            *reinterpret_cast<uint4*>(p.vs_out + dst_off) = vv;
          }
        }
      }
    }
  }

  // ---- teardown ----
  if (MODE == AttnMode::kPrefill && warp < 8 && lane == 0) bulk_wait_all0();  // this warp's TMA stores done
  if (FwdSmem<D, MODE>::kHistStage && warp < 8) cp_async_wait_all();       // staged suffix rows have landed
  tc_fence_before_sync();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag && p.dev_status) atomicOr(p.dev_status, kDevPipelineTimeout);
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace slm
