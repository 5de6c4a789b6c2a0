// Forward kernel, persistent: one CTA per SM takes work items (sequence b,
// q tile qt, head h; longest sequences first) from a device-wide counter in
// list order, and keeps every pipeline running across work items.
//
//   warp 12     producer of Q and K. All 32 lanes build the next item's list
//               of visited kv tiles (from the plan's tile classes) into one of
//               two item slots; lane 0 then loads the item's Q tile and the K
//               tile of every visited kv tile by TMA into a ring of kStages
//               (3 at D=128, 4 at D<=64). K frees after QK^T and Q after the
//               item's last QK^T, so the next item's Q and K arrive while the
//               current item finishes.
//   warp 14     producer of V: the V tile of every visited kv tile into a
//               ring of kStages, each stage freed after its PV. Waiting for V
//               stages never holds back the next item's list, Q and K.
//   warp 13     TMEM owner and MMA issuer (one elected lane):
//                 S[g % 3] = Q K^T             (tcgen05, SMEM x SMEM)
//                 O       += P[g % 3] V        (tcgen05, TMEM x SMEM)
//               with g the tile index counted over all items of the CTA. S
//               runs two tiles ahead of PV, so the tensor core fills one S
//               buffer while the epilogue groups work on the other two. The
//               first PV of an item waits until the epilogue has read out the
//               previous item's O.
//   warps 0-11  epilogue, three groups of four warps: group gr (warps
//               4gr..4gr+3, TMEM lanes 32(w%4)..) takes the tiles with
//               g % 3 == gr, so always S buffer gr. Per tile: P' = S (1 +
//               tanh(alpha S / 2)) (that is silu(alpha S) / N up to the
//               factor alpha / (2N), applied once to O at the store), with
//               the row's interval mask on partial tiles only (full tiles run
//               no mask arithmetic), packed to bf16 in place over the first 64
//               columns of the buffer. At the end of an item two groups
//               each store half of O's columns (bf16, rows past L_b
//               untouched; rows that see no column get zeros) while the
//               group that takes the next item's first tile goes on.
//   warp 15     idle: 16 warps at 128 registers fill the register file, and
//               a third epilogue group hides more TMEM and MUFU latency than
//               two groups at 168 registers.
//
// TMEM (512 columns): S0 [0,128), S1 [128,256), S2 [256,384), O [384, 384+DPV).
// Packed P of buffer b occupies columns [128b, 128b+64).
// SMEM: Q (DPQ/64 chunks of 128 rows x 128 B, 128-byte swizzle), K stages of
// the same shape, V stages of DPV/64 chunks, two item slots.
//
// Template parameters: T the 16-bit input type (bf16 or fp16; P is packed in
// the same type, since one kind::f16 MMA takes one input type), DPQ / DPV
// the head dims of q/k and of v/o rounded up to 64 (32 is a 64-wide box half
// filled with zeros by TMA), NINT the number of func intervals.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace hstu {

// One work item as the producer publishes it to the other roles.
struct FwdItem {
  int b, qt, h, o0, L, nt;
  uint16_t tile[kMaxTiles];  // visited kv tile index | 0x100 if partial
};

template <int DPQ, int DPV>
struct FwdSmem {
  static constexpr int kTileQ = (DPQ / 64) * kBlock * 128;  // bytes of a 128 x DPQ tile
  static constexpr int kTileV = (DPV / 64) * kBlock * 128;  // bytes of a 128 x DPV tile
  static constexpr int kStages = (DPQ == 128 && DPV == 128) ? 3 : 4;  // K/V ring depth
  alignas(1024) uint8_t q[kTileQ];
  alignas(1024) uint8_t k[kStages][kTileQ];
  alignas(1024) uint8_t v[kStages][kTileV];
  alignas(8) uint64_t bar_q_full, bar_q_empty, bar_k_full[kStages], bar_k_empty[kStages],
      bar_v_full[kStages], bar_v_empty[kStages], bar_s_full[3], bar_p_full[3], bar_o_full[2],
      bar_o_empty, bar_item_full[2], bar_item_empty[2], bar_drain;
  uint32_t tmem_base;
  int abort_flag;
  FwdItem item[2];
};

// 227 KB of dynamic shared memory per CTA, with 1 KB of alignment slack.
static_assert(sizeof(FwdSmem<128, 128>) + 1024 <= 232448, "forward shared memory over the per-CTA limit");
static_assert(sizeof(FwdSmem<128, 64>) + 1024 <= 232448, "forward shared memory over the per-CTA limit");
static_assert(sizeof(FwdSmem<64, 128>) + 1024 <= 232448, "forward shared memory over the per-CTA limit");

template <typename S>
__device__ __forceinline__ S& fwd_smem_as(uint8_t* raw) {
  return *reinterpret_cast<S*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
}

// Warp-uniform bounded wait.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  const bool ok = mbar_wait(bar, parity, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

// P' = s (1 + tanh(alpha s / 2)) = silu(alpha s) / N / hc for 32 columns,
// packed to 16 pairs of T; MASKED zeroes the columns whose bit is clear.
template <typename T, bool MASKED>
__device__ __forceinline__ void silu_pack32(const uint32_t (&s)[32], uint32_t mask, float half_alpha,
                                            uint32_t (&pk)[16]) {
#pragma unroll
  for (int e = 0; e < 32; e += 2) {
    float p0 = silu_pu(__uint_as_float(s[e]), half_alpha);
    float p1 = silu_pu(__uint_as_float(s[e + 1]), half_alpha);
    if (MASKED) {
      p0 = ((mask >> e) & 1u) ? p0 : 0.0f;
      p1 = ((mask >> (e + 1)) & 1u) ? p1 : 0.0f;
    }
    pk[e / 2] = Elem<T>::pack2(p0, p1);
  }
}

// Epilogue of one S tile for this warp's 32 rows: HALVES = 2 for all 128
// columns, 1 for a tile whose other 64-column half no row sees (its S MMA
// computed the live half alone into the first 64 columns; col0 is that
// half's first column).
template <typename T, int NINT, bool MASKED, int HALVES = 2>
__device__ __forceinline__ void fwd_tile_epilogue(uint32_t sb, int col0, const int (&lo)[NINT],
                                                  const int (&hi)[NINT], float half_alpha) {
#pragma unroll
  for (int hf = 0; hf < HALVES; ++hf) {
    uint32_t a[32], c[32];
    tmem_ld32(sb + hf * 64, a);
    tmem_ld32(sb + hf * 64 + 32, c);
    tmem_ld_wait(a);
    tmem_ld_wait(c);
    uint32_t pa[16], pc[16];
    silu_pack32<T, MASKED>(a, MASKED ? row_mask_word<NINT>(lo, hi, col0 + hf * 64) : 0u, half_alpha, pa);
    silu_pack32<T, MASKED>(c, MASKED ? row_mask_word<NINT>(lo, hi, col0 + hf * 64 + 32) : 0u, half_alpha,
                        pc);
    // Packed over columns [32 hf, 32 hf + 32) of the buffer, which this warp
    // has already read: K-step kk of the PV MMA reads [8kk, 8kk+8).
    tmem_st16(sb + hf * 32, pa);
    tmem_st16(sb + hf * 32 + 16, pc);
  }
}

// 16 warps: 0-11 three epilogue groups, 12 producer, 13 MMA issuer, 14-15
// idle; 128 registers a thread fill the register file.
constexpr int kFwdThreads = 512;

template <typename T, int DPQ, int DPV, int NINT>
__global__ void __launch_bounds__(kFwdThreads, 1) hstu_fwd_kernel(const __grid_constant__ AttnParams p) {
  using Smem = FwdSmem<DPQ, DPV>;
  constexpr int NS = Smem::kStages;
  constexpr int kTileQ = Smem::kTileQ;
  constexpr int kTileV = Smem::kTileV;
  constexpr int kChunkBytes = kBlock * 128;
  extern __shared__ uint8_t smem_raw[];
  Smem& s = fwd_smem_as<Smem>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int32_t* hdr = p.header;
  if (hdr[kHdrErr] != 0) return;
  const bool uniform = hdr[kHdrUniform] != 0;
  const int n_work = hdr[kHdrNFwd] * p.heads;
  if (static_cast<int>(blockIdx.x) >= n_work) {
    if (threadIdx.x == 0 && !uniform) finish_work(p.header, kHdrFwdNext, kHdrFwdDone);
    return;
  }

  if (threadIdx.x == 0) {
    s.abort_flag = 0;
    mbar_init(smem_u32(&s.bar_q_full), 1);
    mbar_init(smem_u32(&s.bar_q_empty), 1);
    for (int i = 0; i < NS; ++i) {
      mbar_init(smem_u32(&s.bar_k_full[i]), 1);
      mbar_init(smem_u32(&s.bar_k_empty[i]), 1);
      mbar_init(smem_u32(&s.bar_v_full[i]), 1);
      mbar_init(smem_u32(&s.bar_v_empty[i]), 1);
    }
    for (int i = 0; i < 3; ++i) {
      mbar_init(smem_u32(&s.bar_s_full[i]), 1);
      mbar_init(smem_u32(&s.bar_p_full[i]), 128);
    }
    // O is final: one barrier per item slot. The groups that read an item's
    // O out change from item to item; a group that skipped the previous
    // items cannot be two phases behind a slot's barrier, because an item
    // is published in its slot only after the read-out of the item two
    // before it.
    for (int i = 0; i < 2; ++i) mbar_init(smem_u32(&s.bar_o_full[i]), 1);
    mbar_init(smem_u32(&s.bar_o_empty), 256);  // the two epilogue groups that read O out
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&s.bar_item_full[i]), 1);
      mbar_init(smem_u32(&s.bar_item_empty[i]), 2 + 384);  // MMA issuer, V producer, epilogue
    }
    mbar_init(smem_u32(&s.bar_drain), 1);
    fence_mbar_init();
  }
  if (warp == 13) {
    tmem_alloc(smem_u32(&s.tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = s.tmem_base;
  const uint32_t tO = tbase + 384;  // O accumulator columns [384, 384 + DPV)
  volatile int* abort_flag = &s.abort_flag;

  if (warp == 12) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {  // descriptors into the TMA unit's cache before the first copy
      tma_prefetch_map(&p.tm_q);
      tma_prefetch_map(&p.tm_k);
      tma_prefetch_map(&p.tm_v);
    }
    int k_last[NS];  // last use of each K stage, -1 if never used
    for (int i = 0; i < NS; ++i) k_last[i] = -1;
    int q_uses = 0;  // items with at least one tile (one Q load each)
    int g = 0;       // tiles issued over all items
    bool ok = true;
    int i = 0;
    for (; ok; ++i) {
      const int slot = i & 1;
      if (i >= 2 && !warp_wait(smem_u32(&s.bar_item_empty[slot]), ((i >> 1) - 1) & 1, abort_flag)) {
        ok = false;
        break;
      }
      // Work is handed out in list order (longest first): by a fixed stride
      // of the grid when all sequences are equally long, else dynamically,
      // so that CTAs finishing early take the remaining items.
      int w = static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x);
      if (!uniform) {
        if (lane == 0) w = fetch_work(p.header, kHdrFwdNext);
        w = __shfl_sync(0xffffffffu, w, 0);
      }
      // No more work (or, in the checked build, a bad list entry): an item
      // with nt = -1 tells the other roles.
      if (w >= n_work || !list_entry_ok(p, p.list[w / p.heads], false)) {
        if (lane == 0) s.item[slot].nt = -1;
        __threadfence_block();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&s.bar_item_full[slot]));
        break;
      }
      const int code = p.list[w / p.heads];
      const int h = w % p.heads;
      const int b = code >> 8, qt = code & 255;
      const int o0 = p.seq_offsets[b];
      const int L = p.seq_offsets[b + 1] - o0;
      const int ntiles_b = (L + kBlock - 1) / kBlock;
      const uint8_t* cls_row = p.cls + (static_cast<size_t>(b) * p.nt + qt) * p.nt;
      FwdItem& it_slot = s.item[slot];
      int n = 0;
      for (int base = 0; base < ntiles_b; base += 32) {
        const int j = base + lane;
        const uint8_t cb = j < ntiles_b ? cls_row[j] : kSkip;
        const uint8_t c = cb & kClassMask;
        const unsigned m = __ballot_sync(0xffffffffu, c != kSkip);
        // entry: kv tile | 0x100 partial | 0x200 / 0x400 its columns 0..63 /
        // 64..127 seen by no row of the q tile
        if (c != kSkip)
          it_slot.tile[n + __popc(m & ((1u << lane) - 1u))] =
              static_cast<uint16_t>(j | (c == kPartial ? 0x100 : 0) | ((cb & kLoKvDead) ? 0x200 : 0) |
                                    ((cb & kHiKvDead) ? 0x400 : 0));
        n += __popc(m);
      }
      if (lane == 0) {
        it_slot.b = b;
        it_slot.qt = qt;
        it_slot.h = h;
        it_slot.o0 = o0;
        it_slot.L = L;
        it_slot.nt = n;
      }
      __threadfence_block();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&s.bar_item_full[slot]));
        if (n > 0) {
          if (q_uses > 0 && !mbar_wait(smem_u32(&s.bar_q_empty), (q_uses - 1) & 1, abort_flag)) ok = false;
          if (ok) {
            mbar_expect_tx(smem_u32(&s.bar_q_full), kTileQ);
            tma_load_4d(smem_u32(s.q), &p.tm_q, smem_u32(&s.bar_q_full), 0, o0 + qt * kBlock, h, 0);
            ++q_uses;
          }
          for (int t = 0; ok && t < n; ++t) {
            const int gg = g + t, st = gg % NS, use = gg / NS;
            if (use > 0 && !mbar_wait(smem_u32(&s.bar_k_empty[st]), (use - 1) & 1, abort_flag)) {
              ok = false;
              break;
            }
            const uint32_t bar = smem_u32(&s.bar_k_full[st]);
            mbar_expect_tx(bar, kTileQ);
            const int row = o0 + (it_slot.tile[t] & 0xff) * kBlock;
            tma_load_4d(smem_u32(s.k[st]), &p.tm_k, bar, 0, row, h, 0);
            k_last[st] = use;
          }
          g += n;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    }
    // Never leave with a copy in flight.
    if (lane == 0) {
      if (q_uses > 0) mbar_wait_drain(smem_u32(&s.bar_q_full), (q_uses - 1) & 1);
      for (int st = 0; st < NS; ++st)
        if (k_last[st] >= 0) mbar_wait_drain(smem_u32(&s.bar_k_full[st]), k_last[st] & 1);
    }
    __syncwarp();
  } else if (warp == 14) {
    // ------------------------------------------------------------ V producer
    // Follows the item slots the Q/K producer publishes and loads the V tile
    // of every visited kv tile; it holds an item slot until its last V load
    // of that item is issued.
    int v_last[NS];  // last use of each V stage, -1 if never used
    for (int i = 0; i < NS; ++i) v_last[i] = -1;
    int g = 0;  // tiles over all items
    bool ok = true;
    for (int i = 0; ok; ++i) {
      const int slot = i & 1;
      if (!warp_wait(smem_u32(&s.bar_item_full[slot]), (i >> 1) & 1, abort_flag)) break;
      const FwdItem& item = s.item[slot];
      const int nt = item.nt;
      if (nt < 0) break;  // no more work
      if (lane == 0) {
        for (int t = 0; t < nt; ++t) {
          const int gg = g + t, st = gg % NS, use = gg / NS;
          if (use > 0 && !mbar_wait(smem_u32(&s.bar_v_empty[st]), (use - 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t bar = smem_u32(&s.bar_v_full[st]);
          mbar_expect_tx(bar, kTileV);
          const int row = item.o0 + (item.tile[t] & 0xff) * kBlock;
          tma_load_4d(smem_u32(s.v[st]), &p.tm_v, bar, 0, row, item.h, 0);
          v_last[st] = use;
        }
        if (ok) mbar_arrive(smem_u32(&s.bar_item_empty[slot]));
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      g += nt;
    }
    if (lane == 0) {  // never leave with a copy in flight
      for (int st = 0; st < NS; ++st)
        if (v_last[st] >= 0) mbar_wait_drain(smem_u32(&s.bar_v_full[st]), v_last[st] & 1);
    }
    __syncwarp();
  } else if (warp == 13) {
    // ------------------------------------------------------------ MMA issuer
    if (elect_one_sync()) {
      constexpr uint32_t idesc_s = idesc_f16kind(128, 128, false, false, Elem<T>::kUmma);
      constexpr uint32_t idesc_s64 = idesc_f16kind(128, 64, false, false, Elem<T>::kUmma);
      constexpr uint32_t idesc_o = idesc_f16kind(128, DPV, false, true, Elem<T>::kUmma);
      // Descriptors are built once; each MMA only advances a start address.
      const uint64_t dq = sdesc_sw128(smem_u32(s.q), 16, 1024);
      const uint64_t dk0 = sdesc_sw128(smem_u32(s.k[0]), 16, 1024);
      const uint64_t dv0 = sdesc_sw128(smem_u32(s.v[0]), kChunkBytes, 1024);
      int g = 0;       // tiles over all items
      int q_uses = 0;  // items with at least one tile
      bool ok = true;
      int i = 0;
      for (; ok; ++i) {
        const int slot = i & 1;
        if (!mbar_wait(smem_u32(&s.bar_item_full[slot]), (i >> 1) & 1, abort_flag)) break;
        const int nt = s.item[slot].nt;
        if (nt < 0) break;  // no more work
        mbar_arrive(smem_u32(&s.bar_item_empty[slot]));
        if (nt == 0) continue;
        if (!mbar_wait(smem_u32(&s.bar_q_full), q_uses & 1, abort_flag)) break;
        tc_fence_after();
        // S runs two tiles ahead of PV: S(g) goes into buffer g % 3, whose
        // previous tile g - 3 was consumed by a PV issued before it.
        for (int t = 0; t <= nt + 1; ++t) {
          if (t < nt) {
            const int gg = g + t, kst = gg % NS, sb = gg % 3;
            if (!mbar_wait(smem_u32(&s.bar_k_full[kst]), (gg / NS) & 1, abort_flag)) { ok = false; break; }
            tc_fence_after();
            const uint64_t dk = sdesc_advance(dk0, kst * kTileQ);
            const uint32_t d_tmem = tbase + sb * 128;
            const int entry = s.item[slot].tile[t];
            if (entry & 0x600) {
              // One live 64-row half of the K tile: an N=64 MMA into the
              // buffer's first 64 columns.
              const uint32_t live = (entry & 0x200) ? 64u * 128u : 0u;
#pragma unroll
              for (int kk = 0; kk < DPQ / 16; ++kk) {
                const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
                umma_ss(d_tmem, sdesc_advance(dq, off), sdesc_advance(dk, off + live), idesc_s64, kk > 0);
              }
            } else {
#pragma unroll
              for (int kk = 0; kk < DPQ / 16; ++kk) {
                const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
                umma_ss(d_tmem, sdesc_advance(dq, off), sdesc_advance(dk, off), idesc_s, kk > 0);
              }
            }
            umma_commit(smem_u32(&s.bar_s_full[sb]));
            umma_commit(smem_u32(&s.bar_k_empty[kst]));  // K stage free once QK^T is done
            if (t == nt - 1) umma_commit(smem_u32(&s.bar_q_empty));  // Q free for the next item
          }
          if (t >= 2) {
            const int pt = t - 2, gg = g + pt, psb = gg % 3, pkst = gg % NS;
            // The wait for the epilogue to have read out the previous item's O
            // (limit p.handoff_limit_ns; 1 ns, set only by a test, gives up at
            // once so that the abort path runs with copies and MMAs in flight).
            if (pt == 0 && q_uses > 0 &&
                (p.handoff_limit_ns <= 1 ||
                 !mbar_wait(smem_u32(&s.bar_o_empty), (q_uses - 1) & 1, abort_flag, p.handoff_limit_ns))) {
              *abort_flag = 1;
              ok = false;  // the previous item's O has not been read out
              break;
            }
            if (!mbar_wait(smem_u32(&s.bar_v_full[pkst]), (gg / NS) & 1, abort_flag) ||
                !mbar_wait(smem_u32(&s.bar_p_full[psb]), (gg / 3) & 1, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t dv = sdesc_advance(dv0, pkst * kTileV);
            const uint32_t a_tmem = tbase + psb * 128;
            const int pentry = s.item[slot].tile[pt];
            if (pentry & 0x600) {
              // The live half's 64 V rows: four K steps.
              const uint32_t live = (pentry & 0x200) ? 64u : 0u;
#pragma unroll
              for (int kk = 0; kk < kBlock / 32; ++kk)
                umma_ts(tO, a_tmem + kk * 8, sdesc_advance(dv, (live + kk * 16) * 128), idesc_o,
                        (pt > 0 || kk > 0) ? 1u : 0u);
            } else {
              umma_ts(tO, a_tmem, dv, idesc_o, pt > 0 ? 1u : 0u);
#pragma unroll
              for (int kk = 1; kk < kBlock / 16; ++kk)
                umma_ts(tO, a_tmem + kk * 8, sdesc_advance(dv, kk * 16 * 128), idesc_o, 1u);
            }
            umma_commit(smem_u32(&s.bar_v_empty[pkst]));
          }
        }
        if (!ok) break;
        umma_commit(smem_u32(&s.bar_o_full[slot]));
        g += nt;
        ++q_uses;
      }
      // Arrives once every MMA issued above has completed (also on abort).
      umma_commit(smem_u32(&s.bar_drain));
      mbar_wait_drain(smem_u32(&s.bar_drain), 0);
    }
    __syncwarp();
  } else if (warp < 12) {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3, grp = warp >> 2;  // three groups of four warps
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const float half_alpha = 0.5f * p.alpha;
    const float out_scale = 0.5f * p.alpha * p.inv_n;  // hc = alpha / (2N)
    const bool wide = wide_rows_ok(p.out0, p.out0, p.out0, p.dim_v, p.dim_v);
    const int r = quarter * 32 + lane;                 // q row within the tile == TMEM lane
    int g = 0;
    int o_cnt[2] = {0, 0};  // items that filled O, per item slot
    bool ok = true;
    int i = 0;
    for (; ok; ++i) {
      const int slot = i & 1;
      if (!warp_wait(smem_u32(&s.bar_item_full[slot]), (i >> 1) & 1, abort_flag)) break;
      const FwdItem& item = s.item[slot];
      if (item.nt < 0) break;  // no more work
      const int nt = item.nt, qt = item.qt, h = item.h, o0 = item.o0, L = item.L;
      const int i_loc = qt * kBlock + r;
      const bool valid = i_loc < L;
      int lo[NINT], hi[NINT];
      const uint32_t active = p.ivmask[static_cast<size_t>(item.b) * p.nt + qt];
      load_row_intervals<NINT>(p.func, p.total, static_cast<int64_t>(o0) + i_loc, L, valid, lo, hi, active);
      // This group takes the tiles with g % 3 == grp, always S buffer grp.
      for (int t = ((grp - g) % 3 + 3) % 3; t < nt; t += 3) {
        const int gg = g + t, sbuf = gg % 3;
        if (!warp_wait(smem_u32(&s.bar_s_full[sbuf]), (gg / 3) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const int tile = item.tile[t];
        const uint32_t sb = tbase + lane_addr + sbuf * 128;
        if (tile & 0x600) {  // a half tile (partial by construction): its live 64 columns
          const int col0 = (tile & 0xff) * kBlock + ((tile & 0x200) ? kBlock / 2 : 0);
          fwd_tile_epilogue<T, NINT, true, 1>(sb, col0, lo, hi, half_alpha);
        } else if (tile & 0x100) {
          fwd_tile_epilogue<T, NINT, true>(sb, (tile & 0xff) * kBlock, lo, hi, half_alpha);
        } else {
          fwd_tile_epilogue<T, NINT, false>(sb, (tile & 0xff) * kBlock, lo, hi, half_alpha);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(smem_u32(&s.bar_p_full[sbuf]));
      }
      if (!ok) break;
      // The group that takes the next item's first tile (global tile index
      // g + nt) goes on at once; the other two read O out, a column half
      // each.
      // Every group counts the items that fill O, whether or not it reads
      // this one out: o_full[slot] completes a phase per such item.
      const int o_phase = o_cnt[slot] & 1;
      if (nt > 0) ++o_cnt[slot];
      const int skip = (g + nt) % 3;
      if (grp == skip) {
        mbar_arrive(smem_u32(&s.bar_item_empty[slot]));
        g += nt;
        continue;
      }
      const int half = (grp - skip + 3) % 3 - 1;  // 0 or 1
      if (nt > 0) {
        if (!warp_wait(smem_u32(&s.bar_o_full[slot]), o_phase, abort_flag)) break;
        tc_fence_after();
      }
      if (*abort_flag) break;
      // O is complete: the MMA thread has read the item's tile list for its
      // last PV, and this group needs only registers from here on, so the
      // slot may take the item after next during the read-out.
      mbar_arrive(smem_u32(&s.bar_item_empty[slot]));
      constexpr int kHalfCols = DPV / 2;
      constexpr int kNc = kHalfCols / 32;
      T* dst = static_cast<T*>(p.out0) + (static_cast<int64_t>(o0 + qt * kBlock + r) * p.heads + h) * p.dim_v;
      uint32_t v32[kNc][32];
      if (nt > 0) {
#pragma unroll
        for (int cc = 0; cc < kNc; ++cc) tmem_ld32(tO + lane_addr + half * kHalfCols + cc * 32, v32[cc]);
#pragma unroll
        for (int cc = 0; cc < kNc; ++cc) tmem_ld_wait(v32[cc]);
      } else {
#pragma unroll
        for (int cc = 0; cc < kNc; ++cc)
#pragma unroll
          for (int e = 0; e < 32; ++e) v32[cc][e] = 0u;
      }
      // O is in registers: the next item's first PV may overwrite it while
      // the rows are stored.
      if (nt > 0) {
        tc_fence_before();
        mbar_arrive(smem_u32(&s.bar_o_empty));
      }
#pragma unroll
      for (int cc = 0; cc < kNc; ++cc) {
        const int col = half * kHalfCols + cc * 32;
        if (valid && col < p.dim_v) store_row32<T>(dst + col, v32[cc], out_scale, wide);
      }
      g += nt;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
  if (threadIdx.x == 0 && s.abort_flag) atomicOr(p.header + kHdrErr, kErrTimeout);
  if (threadIdx.x == 0 && !uniform) finish_work(p.header, kHdrFwdNext, kHdrFwdDone);
}

// Number of SMs of the current device (looked up per call; cheap).
static inline cudaError_t sm_count(int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  return cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
}

template <typename T, int DPQ, int DPV, int NINT>
static cudaError_t launch_fwd_t(const AttnParams& p, int grid_items, cudaStream_t stream) {
  const int smem = static_cast<int>(sizeof(FwdSmem<DPQ, DPV>)) + 1024;
  static std::atomic<uint64_t> configured{0};  // devices with the limit raised
  cudaError_t e0 = ensure_smem_limit(hstu_fwd_kernel<T, DPQ, DPV, NINT>, smem, configured);
  if (e0 != cudaSuccess) return e0;
  const long long work = static_cast<long long>(grid_items) * p.heads;
  if (work <= 0) return cudaSuccess;
  int sms = 0;
  cudaError_t e = sm_count(&sms);
  if (e != cudaSuccess) return e;
  const long long ctas = work < sms ? work : sms;  // persistent: one CTA per SM
  hstu_fwd_kernel<T, DPQ, DPV, NINT><<<static_cast<unsigned>(ctas), kFwdThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

template <typename T, int DPQ, int DPV>
static cudaError_t launch_fwd_dims(const AttnParams& p, int nint, int grid_items, cudaStream_t stream) {
  switch (nint) {
    case 1: return launch_fwd_t<T, DPQ, DPV, 1>(p, grid_items, stream);
    case 2: return launch_fwd_t<T, DPQ, DPV, 2>(p, grid_items, stream);
    case 3: return launch_fwd_t<T, DPQ, DPV, 3>(p, grid_items, stream);
    case 4: return launch_fwd_t<T, DPQ, DPV, 4>(p, grid_items, stream);
    default: return launch_fwd_t<T, DPQ, DPV, 5>(p, grid_items, stream);
  }
}

// Dispatch on the padded head dims (64 for D <= 64, else 128).
template <typename T>
static cudaError_t launch_fwd_typed(const AttnParams& p, int nint, int grid_items, cudaStream_t stream) {
  if (p.dim > 64) {
    return p.dim_v > 64 ? launch_fwd_dims<T, 128, 128>(p, nint, grid_items, stream)
                        : launch_fwd_dims<T, 128, 64>(p, nint, grid_items, stream);
  }
  return p.dim_v > 64 ? launch_fwd_dims<T, 64, 128>(p, nint, grid_items, stream)
                      : launch_fwd_dims<T, 64, 64>(p, nint, grid_items, stream);
}

}  // namespace hstu
