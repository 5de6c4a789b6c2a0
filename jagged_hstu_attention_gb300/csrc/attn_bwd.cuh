// Backward kernel, persistent: one CTA per SM takes work items, in the order
// of one longest-first list whose entries carry a role bit, from a
// device-wide counter; so both roles run side by side, CTAs that finish
// early take the remaining items, and a CTA keeps its pipelines running
// across items of either role.
//
// dK/dV role -- item (sequence b, kv tile kt, head h). K of the tile is
// copied into TMEM and V stays in SMEM; the Q and dO tiles of every q tile
// that visits kt stream through a ring of 64-row halves. Per half (TMEM
// lanes = kv rows):
//     S^T  = K Q^T   (TMEM x SMEM),  dP^T = V dO^T        (SMEM x SMEM)
//     P^T  = silu(alpha S^T)/N,  dS^T = dP^T * silu'(alpha S^T) * alpha/N
//            (masked on partial tiles, both packed bf16 in place over S^T;
//            the common factor alpha/(2N) is applied once at the stores)
//     dV  += P^T dO,  dK += dS^T Q                       (TMEM x SMEM)
// dK and dV accumulate in TMEM across the whole item and are stored once:
// no atomics, fixed order, bitwise repeatable.
//
// dQ role -- item (sequence b, q tile qt, head h). Q and dO arrive in SMEM
// and are copied into TMEM (tcgen05.cp, into the columns the dK/dV role uses
// for dK), so that S and dP read their A operand from TMEM and only the
// streamed K / V half from SMEM (an N=64 MMA with both operands in SMEM is
// bound by shared-memory reads); K and V of every visited kv tile stream.
// Per kv tile (lanes = q rows):
//     S = Q K^T,  dP = dO V^T;  dS = dP * silu'(alpha S) * alpha/N (packed
//     over S);  dQ += dS K.
// This recomputes S and dP once more per visible tile pair (14 D instead of
// 10 D flops per pair) in exchange for a deterministic dQ with no fp32
// workspace and no reduce-add traffic.
//
// Warps: 0-7 epilogue, 8 producer (tile lists into two item slots, TMA
// loads; streamed tiles travel as 64-row halves through a 5-slot ring, each
// slot freed right after its half's accumulating MMAs), 9 TMEM owner and MMA
// issuer. The next item's lists and resident tiles are fetched while the
// current item finishes; its first accumulating MMA waits until the epilogue
// has read out the previous item's accumulators.
//
// TMEM (512 columns): acc0 [0,128) (dV or dQ), acc1 [128,256) (dK, or the
// dQ role's Q and dO), two S slots at 256 and 320, one dP slot at 384 (64
// columns each), and the dK/dV role's K at 448.
//
// Half-step pipeline: every 128-wide tile is handled as two 64-column halves
// ("half-steps", counted globally as v). S(v) and dP(v) are N=64 MMAs; S(v)
// goes to S slot v % 2, dP(v) to the single dP slot. The epilogue warps form
// two groups of four (TMEM lanes 32(w%4)..); group h takes the half-steps with
// v % 2 == h, always S slot h. A group first reads all of dP(v) and releases
// the dP slot, so that dP(v+1) can be computed while it converts; it then
// packs P^T and dS^T (or dS alone) as bf16 over the S columns it has read.
// S/dP of v + 2 are issued right after the accumulating MMAs of v, so a
// group's conversion of v overlaps the tensor work of the next half-step.
// (Three S slots with K in SMEM measured 1.6% slower on DLRM: the dK/dV
// role's S^T with both operands in SMEM is bound by shared-memory reads.)
//
// Partial-tile masks of the dK/dV role are built by transposition inside
// each warp: lane l takes the two q rows of its half's chunks, computes which
// of the warp's 32 kv rows they see from the rows' intervals, and one ballot
// per kv row turns the bits into that row's 32-q-row words. No warp needs
// another's result, and the cost does not depend on the number of intervals,
// so empty padded intervals stay free.
//
// Template parameters: T the 16-bit input type (bf16 or fp16; P and dS are
// packed in the same type), DPQ / DPV the head dims of q/k and of v/dO
// rounded up to 64, NINT the number of func intervals. Resident and streamed
// operands of the q/k width (res0, str0) hold DPQ columns, those of the v/dO
// width (res1, str1) DPV columns: dV accumulates DPV columns, dK and dQ DPQ.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace hstu {

// One work item as the producer publishes it to the other roles.
struct BwdItem {
  int dkdv, b, tile, h, o0, L, nt;
  int nhs;  // streamed 64-row halves (half-steps) of the item: dead halves are left out
  // visiting (dK/dV) or visited (dQ) tile | 0x100 if partial | 0x200 / 0x400
  // if its streamed half 0 / 1 is dead (dK/dV: q rows that see no column of
  // the kv tile; dQ: kv columns no row of the q tile sees)
  uint16_t idx[kMaxTiles];
};

template <int DPQ, int DPV>
struct BwdSmem {
  static constexpr int kTileQ = (DPQ / 64) * kBlock * 128;        // 128 rows of the q/k width
  static constexpr int kTileV = (DPV / 64) * kBlock * 128;        // 128 rows of the v/dO width
  static constexpr int kHalfQ = (DPQ / 64) * (kBlock / 2) * 128;  // 64 rows
  static constexpr int kHalfV = (DPV / 64) * (kBlock / 2) * 128;
  // Streamed half tiles: as many as fit next to the residents (5 at
  // DPQ = DPV = 128), at most 8.
  static constexpr int kFitSlots = (230400 - kTileQ - kTileV) / (kHalfQ + kHalfV);
  static constexpr int kSlots = kFitSlots < 8 ? kFitSlots : 8;
  // dK/dV role: res0 = K, res1 = V, str0 = Q, str1 = dO.
  // dQ role:    res0 = Q, res1 = dO, str0 = K, str1 = V.
  // Streamed tiles travel as 64-row halves through a ring of kSlots, each
  // slot freed as soon as the accumulating MMAs of its half have completed.
  alignas(1024) uint8_t res0[kTileQ];
  alignas(1024) uint8_t res1[kTileV];
  alignas(1024) uint8_t str0[kSlots][kHalfQ];
  alignas(1024) uint8_t str1[kSlots][kHalfV];
  // TMEM slots of 64 columns after the two accumulators: kSSlots for S
  // (packed P/dS are written over them) and kDpSlots for dP. S/dP of step
  // v + kSSlots are issued right after the accumulating MMAs of step v.
  static constexpr int kSSlots = 2;
  static constexpr int kDpSlots = 1;
  // The dK/dV role copies its resident K into TMEM after the S and dP
  // slots (DPQ / 2 columns), so that S^T reads A from TMEM.
  static constexpr int kKCols = 256 + 64 * (kSSlots + kDpSlots);
  static_assert(kKCols + DPQ / 2 <= 512, "TMEM holds 512 columns");
  alignas(8) uint64_t bar_res_full, bar_res_empty, bar_full[kSlots], bar_empty[kSlots],
      bar_s_full[kSSlots], bar_p_full[kSSlots], bar_dp_free[kDpSlots], bar_acc_full, bar_acc_empty,
      bar_item_full[2], bar_item_empty[2], bar_drain;
  uint32_t tmem_base;
  int abort_flag;
  BwdItem item[2];
};

// 227 KB of dynamic shared memory per CTA, with 1 KB of alignment slack.
static_assert(sizeof(BwdSmem<128, 128>) + 1024 <= 232448, "backward shared memory over the per-CTA limit");
static_assert(sizeof(BwdSmem<128, 64>) + 1024 <= 232448, "backward shared memory over the per-CTA limit");
static_assert(sizeof(BwdSmem<64, 128>) + 1024 <= 232448, "backward shared memory over the per-CTA limit");
static_assert(sizeof(BwdSmem<64, 64>) + 1024 <= 232448, "backward shared memory over the per-CTA limit");
static_assert(BwdSmem<128, 128>::kSlots == 5, "five streamed slots at D = 128");

template <typename S>
__device__ __forceinline__ S& smem_as_b(uint8_t* raw) {
  return *reinterpret_cast<S*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ bool warp_wait_b(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  const bool ok = mbar_wait(bar, parity, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

// Reads NC 32-column accumulator chunks (TMEM addresses ta[c], this warp's
// lanes) with a single wait, or zeros when `have` is false.
template <int NC>
__device__ __forceinline__ void load_acc_chunks(const uint32_t (&ta)[NC], bool have, uint32_t (&a)[NC][32]) {
  if (have) {
#pragma unroll
    for (int c = 0; c < NC; ++c) tmem_ld32(ta[c], a[c]);
#pragma unroll
    for (int c = 0; c < NC; ++c) tmem_ld_wait(a[c]);
  } else {
#pragma unroll
    for (int c = 0; c < NC; ++c)
#pragma unroll
      for (int e = 0; e < 32; ++e) a[c][e] = 0u;
  }
}

// Writes chunk c of `a`, times `scale`, as columns [col[c], col[c] + 32) of
// the row dst[c] of dim[c] elements (nothing for an invalid row or columns
// past dim[c]).
template <typename T, int NC>
__device__ __forceinline__ void store_acc_chunks(const uint32_t (&a)[NC][32], T* const (&dst)[NC],
                                                 const int (&col)[NC], const int (&dim)[NC], bool valid,
                                                 float scale, bool wide) {
#pragma unroll
  for (int c = 0; c < NC; ++c)
    if (valid && col[c] < dim[c]) store_row32<T>(dst[c] + col[c], a[c], scale, wide);
}

// 16 columns [C0, C0 + 16) of 32 loaded S and dP columns -> packed T
// P' = s (1 + t) (when WANT_P) and G' = dP (1 + t)(1 + h - h t), h = alpha s / 2,
// t = tanh(h): the backward quantities up to the factor alpha / (2N) applied
// to dV, dK and dQ at their store. MASKED zeroes the columns whose bit (of
// the 32-column word) is clear.
template <typename T, int C0, bool MASKED, bool WANT_P>
__device__ __forceinline__ void epilogue16(const uint32_t (&sv)[32], const uint32_t (&dv)[32],
                                           uint32_t mask, float half_alpha, uint32_t (&pp)[8],
                                           uint32_t (&pd)[8]) {
#pragma unroll
  for (int e = 0; e < 16; e += 2) {
    float g[2], pv[2];
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      const float sc = __uint_as_float(sv[C0 + e + x]);
      const float dp = __uint_as_float(dv[C0 + e + x]);
      if (WANT_P) silu_pu_gu(sc, dp, half_alpha, pv[x], g[x]);
      else g[x] = silu_gu(sc, dp, half_alpha);
      if (MASKED) {
        const bool on = (mask >> (C0 + e + x)) & 1u;
        if (WANT_P) pv[x] = on ? pv[x] : 0.0f;
        g[x] = on ? g[x] : 0.0f;
      }
    }
    if (WANT_P) pp[e / 2] = Elem<T>::pack2(pv[0], pv[1]);
    pd[e / 2] = Elem<T>::pack2(g[0], g[1]);
  }
}

// Converts one 32-column chunk (the q rows of K-steps 2c and 2c + 1 of a
// half) and packs it over S columns this warp has already read. dK/dV role:
// K-step ks of the accumulating MMAs reads P^T from slot columns
// [16ks, 16ks + 8) and dS^T from [16ks + 8, 16ks + 16); dQ role: dS from
// [8ks, 8ks + 8).
template <typename T, bool MASKED, bool DKDV>
__device__ __forceinline__ void convert_chunk(const uint32_t (&sv)[32], const uint32_t (&dv)[32],
                                              uint32_t mask, float half_alpha, uint32_t xs, int c) {
  uint32_t pp[8], pd[8];
  epilogue16<T, 0, MASKED, DKDV>(sv, dv, mask, half_alpha, pp, pd);
  if (DKDV) tmem_st8x2(xs + 32 * c, pp, pd);
  else tmem_st8(xs + 16 * c, pd);
  epilogue16<T, 16, MASKED, DKDV>(sv, dv, mask, half_alpha, pp, pd);
  if (DKDV) tmem_st8x2(xs + 32 * c + 16, pp, pd);
  else tmem_st8(xs + 16 * c + 8, pd);
}

template <typename T, int DPQ, int DPV, int NINT>
__global__ void __launch_bounds__(320, 1) hstu_bwd_kernel(const __grid_constant__ AttnParams p) {
  using Smem = BwdSmem<DPQ, DPV>;
  constexpr int kChunkBytes = kBlock * 128;       // one 64-column chunk of a 128-row tile
  constexpr int kHalfChunk = (kBlock / 2) * 128;  // one 64-column chunk of a 64-row half
  extern __shared__ uint8_t smem_raw[];
  Smem& s = smem_as_b<Smem>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int32_t* hdr = p.header;
  if (hdr[kHdrErr] != 0) return;
  const bool uniform = hdr[kHdrUniform] != 0;
  const int n_work = hdr[kHdrNBwd] * p.heads;
  if (static_cast<int>(blockIdx.x) >= n_work) {
    if (threadIdx.x == 0 && !uniform) finish_work(p.header, kHdrBwdNext, kHdrBwdDone);
    return;
  }

  if (threadIdx.x == 0) {
    s.abort_flag = 0;
    mbar_init(smem_u32(&s.bar_res_full), 1);
    mbar_init(smem_u32(&s.bar_res_empty), 1);
    for (int i = 0; i < Smem::kSlots; ++i) {
      mbar_init(smem_u32(&s.bar_full[i]), 1);
      mbar_init(smem_u32(&s.bar_empty[i]), 1);
    }
    for (int i = 0; i < Smem::kSSlots; ++i) {
      mbar_init(smem_u32(&s.bar_s_full[i]), 1);
      mbar_init(smem_u32(&s.bar_p_full[i]), 128);
    }
    for (int i = 0; i < Smem::kDpSlots; ++i) mbar_init(smem_u32(&s.bar_dp_free[i]), 128);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&s.bar_item_full[i]), 1);
      mbar_init(smem_u32(&s.bar_item_empty[i]), 1 + 256);  // MMA issuer + epilogue threads
    }
    mbar_init(smem_u32(&s.bar_acc_full), 1);
    mbar_init(smem_u32(&s.bar_acc_empty), 256);
    mbar_init(smem_u32(&s.bar_drain), 1);
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(&s.tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = s.tmem_base;
  const uint32_t t_acc0 = tbase;        // dV (dK/dV role) or dQ (dQ role)
  const uint32_t t_acc1 = tbase + 128;  // dK (dK/dV role)
  const uint32_t tS = tbase + 256;      // S slot k at tS + 64 k
  const uint32_t tdP = tS + 64 * Smem::kSSlots;  // dP slot j at tdP + 64 j
  const uint32_t tK = tbase + Smem::kKCols;       // dK/dV role: resident K
  volatile int* abort_flag = &s.abort_flag;
  const size_t nt_all = static_cast<size_t>(p.nt);

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {  // descriptors into the TMA unit's cache before the first copy
      tma_prefetch_map(&p.tm_q);
      tma_prefetch_map(&p.tm_k);
      tma_prefetch_map(&p.tm_v);
      tma_prefetch_map(&p.tm_do);
      tma_prefetch_map(&p.tm_q64);
      tma_prefetch_map(&p.tm_k64);
      tma_prefetch_map(&p.tm_v64);
      tma_prefetch_map(&p.tm_do64);
    }
    int str_last[Smem::kSlots];  // last use of each ring slot, -1 if never used
    for (int st = 0; st < Smem::kSlots; ++st) str_last[st] = -1;
    int res_uses = 0;  // items with at least one tile (one resident load each)
    int ghs = 0;       // streamed halves over all items
    bool ok = true;
    int i = 0;
    for (; ok; ++i) {
      const int slot = i & 1;
      if (i >= 2 && !warp_wait_b(smem_u32(&s.bar_item_empty[slot]), ((i >> 1) - 1) & 1, abort_flag)) {
        ok = false;
        break;
      }
      // Work is handed out in list order (longest first): by a fixed stride
      // of the grid when all sequences are equally long, else dynamically,
      // so that CTAs finishing early take the remaining items.
      int w = static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x);
      if (!uniform) {
        if (lane == 0) w = fetch_work(p.header, kHdrBwdNext);
        w = __shfl_sync(0xffffffffu, w, 0);
      }
      // No more work (or, in the checked build, a bad list entry): an item
      // with nt = -1 tells the other roles.
      if (w >= n_work || !list_entry_ok(p, p.list[w / p.heads], true)) {
        if (lane == 0) s.item[slot].nt = -1;
        __threadfence_block();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&s.bar_item_full[slot]));
        break;
      }
      const int code = p.list[w / p.heads];
      const int h = w % p.heads;
      const bool dkdv = (code & kRoleDkdv) != 0;
      const int b = (code & ~kRoleDkdv) >> 8, tile = code & 255;
      const int o0 = p.seq_offsets[b];
      const int L = p.seq_offsets[b + 1] - o0;
      const int ntiles_b = (L + kBlock - 1) / kBlock;
      const uint8_t* cls_b = p.cls + static_cast<size_t>(b) * nt_all * nt_all;
      BwdItem& it_slot = s.item[slot];
      // dK/dV: q tiles visiting kv tile `tile` (a column of the class matrix);
      // dQ: kv tiles visited by q tile `tile` (a row of it).
      int n = 0, nhs = 0;
      for (int base = 0; base < ntiles_b; base += 32) {
        const int x = base + lane;
        uint8_t cb = kSkip;
        if (x < ntiles_b)
          cb = dkdv ? cls_b[static_cast<size_t>(x) * nt_all + tile] : cls_b[static_cast<size_t>(tile) * nt_all + x];
        const uint8_t c = cb & kClassMask;
        const int dead0 = (cb & (dkdv ? kLoQDead : kLoKvDead)) ? 1 : 0;
        const int dead1 = (cb & (dkdv ? kHiQDead : kHiKvDead)) ? 1 : 0;
        const unsigned m = __ballot_sync(0xffffffffu, c != kSkip);
        if (c != kSkip)
          it_slot.idx[n + __popc(m & ((1u << lane) - 1u))] =
              static_cast<uint16_t>(x | (c == kPartial ? 0x100 : 0) | (dead0 << 9) | (dead1 << 10));
        n += __popc(m);
        nhs += __reduce_add_sync(0xffffffffu, c != kSkip ? 2 - dead0 - dead1 : 0);
      }
      if (lane == 0) {
        it_slot.dkdv = dkdv ? 1 : 0;
        it_slot.b = b;
        it_slot.tile = tile;
        it_slot.h = h;
        it_slot.o0 = o0;
        it_slot.L = L;
        it_slot.nt = n;
        it_slot.nhs = nhs;
      }
      __threadfence_block();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&s.bar_item_full[slot]));
        if (n > 0) {
          const CUtensorMap* m_res0 = dkdv ? &p.tm_k : &p.tm_q;
          const CUtensorMap* m_res1 = dkdv ? &p.tm_v : &p.tm_do;
          const CUtensorMap* m_str0 = dkdv ? &p.tm_q64 : &p.tm_k64;
          const CUtensorMap* m_str1 = dkdv ? &p.tm_do64 : &p.tm_v64;
          if (res_uses > 0 && !mbar_wait(smem_u32(&s.bar_res_empty), (res_uses - 1) & 1, abort_flag))
            ok = false;
          if (ok) {
            const uint32_t br = smem_u32(&s.bar_res_full);
            mbar_expect_tx(br, Smem::kTileQ + Smem::kTileV);
            const int row0 = o0 + tile * kBlock;
            tma_load_4d(smem_u32(s.res0), m_res0, br, 0, row0, h, 0);
            tma_load_4d(smem_u32(s.res1), m_res1, br, 0, row0, h, 0);
            ++res_uses;
          }
          for (int t = 0; ok && t < 2 * n; ++t) {  // 64-row halves that are not dead
            const int e = it_slot.idx[t >> 1];
            if (e & (0x200 << (t & 1))) continue;
            const int gh = ghs++, st = gh % Smem::kSlots, use = gh / Smem::kSlots;
            if (use > 0 && !mbar_wait(smem_u32(&s.bar_empty[st]), (use - 1) & 1, abort_flag)) {
              ok = false;
              break;
            }
            const int srow0 = o0 + (e & 0xff) * kBlock + (t & 1) * (kBlock / 2);
            const uint32_t bar = smem_u32(&s.bar_full[st]);
            mbar_expect_tx(bar, Smem::kHalfQ + Smem::kHalfV);
            tma_load_4d(smem_u32(s.str0[st]), m_str0, bar, 0, srow0, h, 0);
            tma_load_4d(smem_u32(s.str1[st]), m_str1, bar, 0, srow0, h, 0);
            str_last[st] = use;
          }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    }
    // Never leave with a copy in flight.
    if (lane == 0) {
      if (res_uses > 0) mbar_wait_drain(smem_u32(&s.bar_res_full), (res_uses - 1) & 1);
      for (int st = 0; st < Smem::kSlots; ++st)
        if (str_last[st] >= 0) mbar_wait_drain(smem_u32(&s.bar_full[st]), str_last[st] & 1);
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (elect_one_sync()) {
      // Half-step pipeline: step v covers the 64-column half (v & 1) of tile
      // v >> 1. S/dP run kSSlots steps ahead of the accumulating MMAs.
      constexpr uint32_t idesc_s = idesc_f16kind(128, 64, false, false, Elem<T>::kUmma);
      // dV accumulates DPV columns (B = dO); dK and dQ DPQ columns (B = Q or K).
      constexpr uint32_t idesc_accv = idesc_f16kind(128, DPV, false, true, Elem<T>::kUmma);
      constexpr uint32_t idesc_accq = idesc_f16kind(128, DPQ, false, true, Elem<T>::kUmma);
      // Descriptors are built once; each MMA only advances a start address.
      const uint64_t dr0 = sdesc_sw128(smem_u32(s.res0), 16, 1024);
      const uint64_t dr1 = sdesc_sw128(smem_u32(s.res1), 16, 1024);
      const uint64_t ds0 = sdesc_sw128(smem_u32(s.str0[0]), 16, 1024);
      const uint64_t ds1 = sdesc_sw128(smem_u32(s.str1[0]), 16, 1024);
      const uint64_t ds0_mn = sdesc_sw128(smem_u32(s.str0[0]), kHalfChunk, 1024);
      const uint64_t ds1_mn = sdesc_sw128(smem_u32(s.str1[0]), kHalfChunk, 1024);
      // dQ role: Q and dO are copied into TMEM (the columns a dK/dV item
      // uses for dK), so that its S and dP MMAs read A from TMEM and only the
      // streamed K / V half from shared memory. With both operands in shared
      // memory an N=64 MMA is bound by shared-memory reads.
      const uint32_t tQr = t_acc1, tdOr = t_acc1 + DPQ / 2;
      // The wait for the epilogue to have read out the previous item's
      // accumulators (limit p.handoff_limit_ns; a limit of 1 ns, set only by
      // a test, gives up at once so that the abort path runs with this
      // item's copies and MMAs in flight).
      auto handoff_wait = [&](uint32_t bar, uint32_t parity) -> bool {
        if (p.handoff_limit_ns <= 1) {
          *abort_flag = 1;
          return false;
        }
        return mbar_wait(bar, parity, abort_flag, p.handoff_limit_ns);
      };
      int ghs = 0;       // half-steps over all items
      int res_uses = 0;  // items with at least one tile
      bool prev_dkdv = false;  // role of the previous item with at least one tile
      bool ok = true;
      int i = 0;
      for (; ok; ++i) {
        const int slot = i & 1;
        if (!mbar_wait(smem_u32(&s.bar_item_full[slot]), (i >> 1) & 1, abort_flag)) break;
        const int nt = s.item[slot].nt;
        if (nt < 0) break;  // no more work
        const bool dkdv = s.item[slot].dkdv != 0;
        const int nsteps = s.item[slot].nhs;  // every field this thread reads, before the slot is released
        mbar_arrive(smem_u32(&s.bar_item_empty[slot]));
        if (nt == 0) continue;
        if (!mbar_wait(smem_u32(&s.bar_res_full), res_uses & 1, abort_flag)) break;
        tc_fence_after();
        if (!dkdv) {
          // The copy overwrites the dK columns: after a dK/dV item, wait until
          // the epilogue has read them out. (After a dQ item the columns hold
          // its Q and dO, whose last readers -- its S/dP MMAs -- completed
          // before its last accumulating MMA was issued.)
          if (res_uses > 0 && prev_dkdv && !handoff_wait(smem_u32(&s.bar_acc_empty), (res_uses - 1) & 1))
            break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < DPQ / 16; ++kk)
            tmem_cp_128x256b(tQr + 8 * kk, sdesc_advance(dr0, (kk >> 2) * kChunkBytes + (kk & 3) * 32));
#pragma unroll
          for (int kk = 0; kk < DPV / 16; ++kk)
            tmem_cp_128x256b(tdOr + 8 * kk, sdesc_advance(dr1, (kk >> 2) * kChunkBytes + (kk & 3) * 32));
          umma_commit(smem_u32(&s.bar_res_empty));  // shared-memory residents free once copied
        } else {
          // K into TMEM for S^T = K Q^T. Its previous readers, the S MMAs of
          // the previous dK/dV item, completed before that item's last
          // accumulating MMAs were issued.
#pragma unroll
          for (int kk = 0; kk < DPQ / 16; ++kk)
            tmem_cp_128x256b(tK + 8 * kk, sdesc_advance(dr0, (kk >> 2) * kChunkBytes + (kk & 3) * 32));
        }
        const int gv0 = ghs;  // global index of this item's first half-step
        // S/dP of step v (N = 64 MMAs): S (or S^T) = res0 . str0_h^T into S
        // slot gv % kSSlots, dP (or dP^T) = res1 . str1_h^T into the dP slot
        // once the epilogue has read dP of step gv - 1 out of it.
        auto issue_sdp = [&](int v) -> bool {
          const int gv = gv0 + v, st = gv % Smem::kSlots, k = gv % Smem::kSSlots, j = gv % Smem::kDpSlots;
          if (!mbar_wait(smem_u32(&s.bar_full[st]), (gv / Smem::kSlots) & 1, abort_flag)) return false;
          tc_fence_after();
          const uint64_t b0 = sdesc_advance(ds0, st * Smem::kHalfQ), b1 = sdesc_advance(ds1, st * Smem::kHalfV);
          if (dkdv) {
#pragma unroll
            for (int kk = 0; kk < DPQ / 16; ++kk) {
              const uint32_t boff = (kk >> 2) * kHalfChunk + (kk & 3) * 32;
              umma_ts(tS + 64 * k, tK + 8 * kk, sdesc_advance(b0, boff), idesc_s, kk > 0);
            }
          } else {
#pragma unroll
            for (int kk = 0; kk < DPQ / 16; ++kk) {
              const uint32_t boff = (kk >> 2) * kHalfChunk + (kk & 3) * 32;
              umma_ts(tS + 64 * k, tQr + 8 * kk, sdesc_advance(b0, boff), idesc_s, kk > 0);
            }
          }
          // dP slot j is free once the epilogue has read out dP of step gv - kDpSlots.
          if (gv >= Smem::kDpSlots &&
              !mbar_wait(smem_u32(&s.bar_dp_free[j]), ((gv - Smem::kDpSlots) / Smem::kDpSlots) & 1, abort_flag))
            return false;
          tc_fence_after();
          if (dkdv) {
#pragma unroll
            for (int kk = 0; kk < DPV / 16; ++kk) {
              const uint32_t aoff = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
              const uint32_t boff = (kk >> 2) * kHalfChunk + (kk & 3) * 32;
              umma_ss(tdP + 64 * j, sdesc_advance(dr1, aoff), sdesc_advance(b1, boff), idesc_s, kk > 0);
            }
          } else {
#pragma unroll
            for (int kk = 0; kk < DPV / 16; ++kk) {
              const uint32_t boff = (kk >> 2) * kHalfChunk + (kk & 3) * 32;
              umma_ts(tdP + 64 * j, tdOr + 8 * kk, sdesc_advance(b1, boff), idesc_s, kk > 0);
            }
          }
          umma_commit(smem_u32(&s.bar_s_full[k]));
          if (dkdv && v == nsteps - 1) umma_commit(smem_u32(&s.bar_res_empty));  // residents free
          return true;
        };
        // S of step v + kSSlots reuses the S slot of step v, whose packed
        // P/dS the accumulating MMAs of step v (issued just before, in order)
        // read.
        for (int v = 0; ok && v < Smem::kSSlots && v < nsteps; ++v) ok = issue_sdp(v);
        for (int v = 0; ok && v < nsteps; ++v) {
          const int gv = gv0 + v, pst = gv % Smem::kSlots, k = gv % Smem::kSSlots;
          if (v == 0 && res_uses > 0 && !handoff_wait(smem_u32(&s.bar_acc_empty), (res_uses - 1) & 1)) {
            ok = false;  // the previous item's accumulators have not been read out
            break;
          }
          if (!mbar_wait(smem_u32(&s.bar_p_full[k]), (gv / Smem::kSSlots) & 1, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t m0 = sdesc_advance(ds0_mn, pst * Smem::kHalfQ);
          const uint64_t m1 = sdesc_advance(ds1_mn, pst * Smem::kHalfV);
          const uint32_t first = v > 0 ? 1u : 0u;
          const uint32_t xs = tS + 64 * k;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {  // K = the 64 rows of this half
            const uint32_t acc = ks > 0 ? 1u : first;
            if (dkdv) {
              // dV += P^T dO (dO = str1, MN-major); dK += dS^T Q (Q = str0, MN-major)
              umma_ts(t_acc0, xs + 16 * ks, sdesc_advance(m1, ks * 16 * 128), idesc_accv, acc);
              umma_ts(t_acc1, xs + 16 * ks + 8, sdesc_advance(m0, ks * 16 * 128), idesc_accq, acc);
            } else {
              // dQ += dS K (K = str0, MN-major)
              umma_ts(t_acc0, xs + 8 * ks, sdesc_advance(m0, ks * 16 * 128), idesc_accq, acc);
            }
          }
          umma_commit(smem_u32(&s.bar_empty[pst]));  // this half's slot is free
          if (v + Smem::kSSlots < nsteps && !issue_sdp(v + Smem::kSSlots)) ok = false;
        }
        if (!ok) break;
        umma_commit(smem_u32(&s.bar_acc_full));
        ghs += nsteps;
        ++res_uses;
        prev_dkdv = dkdv;
      }
      // Arrives once every MMA issued above has completed (also on abort).
      umma_commit(smem_u32(&s.bar_drain));
      mbar_wait_drain(smem_u32(&s.bar_drain), 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3, half = warp >> 2;
    const int r = quarter * 32 + lane;  // TMEM lane: kv row (dK/dV role) or q row (dQ role)
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const float half_alpha = 0.5f * p.alpha;
    const float out_scale = 0.5f * p.alpha * p.inv_n;  // hc = alpha / (2N)
    // 32-byte stores need every output row to start on a 32-byte boundary.
    const bool wide = wide_rows_ok(p.out0, p.out1, p.out2, p.dim, p.dim_v);
    const int hh = half;  // this warp group takes the half-steps whose global index has parity hh
    int g0 = 0;           // half-steps over all items
    int acc_uses = 0;
    bool ok = true;
    int i = 0;
    for (; ok; ++i) {
      const int slot = i & 1;
      if (!warp_wait_b(smem_u32(&s.bar_item_full[slot]), (i >> 1) & 1, abort_flag)) break;
      const BwdItem& item = s.item[slot];
      if (item.nt < 0) break;  // no more work
      const bool dkdv = item.dkdv != 0;
      const int nt = item.nt, tile = item.tile, h = item.h, o0 = item.o0, L = item.L;
      const int own_loc = tile * kBlock + r;
      const bool valid = own_loc < L;
      int lo[NINT], hi[NINT];
      const uint8_t* iv_b = p.ivmask + static_cast<size_t>(item.b) * nt_all;
      if (!dkdv)
        load_row_intervals<NINT>(p.func, p.total, static_cast<int64_t>(o0) + own_loc, L, valid, lo, hi,
                                 iv_b[tile]);
      // Walk the item's half-steps in order (dead halves are not streamed);
      // this group takes those with an odd or even global index, hh.
      int lhs = 0;  // half-steps of this item so far
      for (int hs_t = 0; ok && hs_t < 2 * nt; ++hs_t) {
        const int it = hs_t >> 1, hsel = hs_t & 1;  // tile entry and its half
        const int e = item.idx[it];
        if (e & (0x200 << hsel)) continue;  // dead half
        const int gv = g0 + lhs++;          // global half-step
        if ((gv & 1) != hh) continue;       // the other group's
        const int other = e & 0xff;
        const bool partial = (e & 0x100) != 0;
        uint32_t qmask0 = 0, qmask1 = 0;
        if (dkdv && partial) {
          // Lane l takes q rows 64 hsel + l and 64 hsel + 32 + l of the
          // visiting q tile and finds which of this warp's 32 kv rows each of
          // them sees; one ballot per kv row turns the bits around, so that
          // lane j holds the q-row masks of kv row 32 quarter + j for both
          // chunks of the half.
          int flo[NINT], fhi[NINT];
          const int qa = other * kBlock + 64 * hsel + lane;
          const int kv0 = tile * kBlock + 32 * quarter;
          load_row_intervals<NINT>(p.func, p.total, static_cast<int64_t>(o0) + qa, L, qa < L, flo, fhi,
                                   iv_b[other]);
          const uint32_t w0 = row_mask_word<NINT>(flo, fhi, kv0);
          load_row_intervals<NINT>(p.func, p.total, static_cast<int64_t>(o0) + qa + 32, L, qa + 32 < L, flo,
                                   fhi, iv_b[other]);
          const uint32_t w1 = row_mask_word<NINT>(flo, fhi, kv0);
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const uint32_t b0 = __ballot_sync(0xffffffffu, (w0 >> j) & 1u);
            const uint32_t b1 = __ballot_sync(0xffffffffu, (w1 >> j) & 1u);
            if (lane == j) {
              qmask0 = b0;
              qmask1 = b1;
            }
          }
        }
        const int k = gv % Smem::kSSlots, j = gv % Smem::kDpSlots;
        const uint32_t xs = tS + 64 * k + lane_addr;
        if (!warp_wait_b(smem_u32(&s.bar_s_full[k]), (gv / Smem::kSSlots) & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // All of dP first, so that the dP slot is released for the next step.
        uint32_t dv0[32], dv1[32], sv[32];
        tmem_ld32(tdP + 64 * j + lane_addr, dv0);
        tmem_ld32(tdP + 64 * j + lane_addr + 32, dv1);
        tmem_ld32(xs, sv);
        tmem_ld_wait(dv0);
        tmem_ld_wait(dv1);
        tmem_ld_wait(sv);
        tc_fence_before();
        mbar_arrive(smem_u32(&s.bar_dp_free[j]));
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int chunk = 2 * hsel + c;  // 32-column chunk of the tile's 128
          if (c == 1) {
            tmem_ld32(xs + 32, sv);
            tmem_ld_wait(sv);
          }
          const uint32_t(&dv)[32] = c == 0 ? dv0 : dv1;
          if (partial) {  // item-uniform: full tiles run no mask arithmetic
            const uint32_t mask = dkdv ? (c == 0 ? qmask0 : qmask1)
                                       : row_mask_word<NINT>(lo, hi, other * kBlock + chunk * 32);
            if (dkdv) convert_chunk<T, true, true>(sv, dv, mask, half_alpha, xs, c);
            else convert_chunk<T, true, false>(sv, dv, mask, half_alpha, xs, c);
          } else {
            if (dkdv) convert_chunk<T, false, true>(sv, dv, 0u, half_alpha, xs, c);
            else convert_chunk<T, false, false>(sv, dv, 0u, half_alpha, xs, c);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(smem_u32(&s.bar_p_full[k]));
      }
      if (!ok) break;
      // The item's fields are in registers from here on: its slot may take
      // the item after next while the accumulators are read out.
      mbar_arrive(smem_u32(&s.bar_item_empty[slot]));
      if (nt > 0) {
        if (!warp_wait_b(smem_u32(&s.bar_acc_full), acc_uses & 1, abort_flag)) break;
        tc_fence_after();
      }
      if (*abort_flag) break;
      const int64_t row = static_cast<int64_t>(o0 + own_loc) * p.heads + h;
      // This warp's half of the accumulators (dV and dK, or dQ) is loaded
      // with one wait and released before the rows are stored, so that the
      // next item may overwrite those columns meanwhile.
      if (dkdv) {
        constexpr int kV = DPV / 64, kQ = DPQ / 64;  // chunks per half of dV / dK
        uint32_t ta[kV + kQ];
        T* dst[kV + kQ];
        int col[kV + kQ], dim[kV + kQ];
#pragma unroll
        for (int c = 0; c < kV; ++c) {
          col[c] = half * (DPV / 2) + 32 * c;
          ta[c] = t_acc0 + lane_addr + col[c];
          dst[c] = static_cast<T*>(p.out2) + row * p.dim_v;
          dim[c] = p.dim_v;
        }
#pragma unroll
        for (int c = 0; c < kQ; ++c) {
          col[kV + c] = half * (DPQ / 2) + 32 * c;
          ta[kV + c] = t_acc1 + lane_addr + col[kV + c];
          dst[kV + c] = static_cast<T*>(p.out1) + row * p.dim;
          dim[kV + c] = p.dim;
        }
        uint32_t a[kV + kQ][32];
        load_acc_chunks<kV + kQ>(ta, nt > 0, a);
        if (nt > 0) {
          tc_fence_before();
          mbar_arrive(smem_u32(&s.bar_acc_empty));
          ++acc_uses;
        }
        store_acc_chunks<T, kV + kQ>(a, dst, col, dim, valid, out_scale, wide);
      } else {
        constexpr int kC = DPQ / 64;  // chunks per half of dQ
        uint32_t ta[kC];
        T* dst[kC];
        int col[kC], dim[kC];
#pragma unroll
        for (int c = 0; c < kC; ++c) {
          col[c] = half * (DPQ / 2) + 32 * c;
          ta[c] = t_acc0 + lane_addr + col[c];
          dst[c] = static_cast<T*>(p.out0) + row * p.dim;
          dim[c] = p.dim;
        }
        uint32_t a[kC][32];
        load_acc_chunks<kC>(ta, nt > 0, a);
        if (nt > 0) {
          tc_fence_before();
          mbar_arrive(smem_u32(&s.bar_acc_empty));
          ++acc_uses;
        }
        store_acc_chunks<T, kC>(a, dst, col, dim, valid, out_scale, wide);
      }
      g0 += lhs;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
  if (threadIdx.x == 0 && s.abort_flag) atomicOr(p.header + kHdrErr, kErrTimeout);
  if (threadIdx.x == 0 && !uniform) finish_work(p.header, kHdrBwdNext, kHdrBwdDone);
}

template <typename T, int DPQ, int DPV, int NINT>
static cudaError_t launch_bwd_t(const AttnParams& p, int grid_items, cudaStream_t stream) {
  const int smem = static_cast<int>(sizeof(BwdSmem<DPQ, DPV>)) + 1024;
  static std::atomic<uint64_t> configured{0};  // devices with the limit raised
  cudaError_t e0 = ensure_smem_limit(hstu_bwd_kernel<T, DPQ, DPV, NINT>, smem, configured);
  if (e0 != cudaSuccess) return e0;
  const long long work = 2LL * grid_items * p.heads;
  if (work <= 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long long ctas = work < sms ? work : sms;  // persistent: one CTA per SM
  hstu_bwd_kernel<T, DPQ, DPV, NINT><<<static_cast<unsigned>(ctas), 320, smem, stream>>>(p);
  return cudaGetLastError();
}

template <typename T, int DPQ, int DPV>
static cudaError_t launch_bwd_dims(const AttnParams& p, int nint, int grid_items, cudaStream_t stream) {
  switch (nint) {
    case 1: return launch_bwd_t<T, DPQ, DPV, 1>(p, grid_items, stream);
    case 2: return launch_bwd_t<T, DPQ, DPV, 2>(p, grid_items, stream);
    case 3: return launch_bwd_t<T, DPQ, DPV, 3>(p, grid_items, stream);
    case 4: return launch_bwd_t<T, DPQ, DPV, 4>(p, grid_items, stream);
    default: return launch_bwd_t<T, DPQ, DPV, 5>(p, grid_items, stream);
  }
}

// Dispatch on the padded head dims (64 for D <= 64, else 128).
template <typename T>
static cudaError_t launch_bwd_typed(const AttnParams& p, int nint, int grid_items, cudaStream_t stream) {
  if (p.dim > 64) {
    return p.dim_v > 64 ? launch_bwd_dims<T, 128, 128>(p, nint, grid_items, stream)
                        : launch_bwd_dims<T, 128, 64>(p, nint, grid_items, stream);
  }
  return p.dim_v > 64 ? launch_bwd_dims<T, 64, 128>(p, nint, grid_items, stream)
                      : launch_bwd_dims<T, 64, 64>(p, nint, grid_items, stream);
}

}  // namespace hstu
