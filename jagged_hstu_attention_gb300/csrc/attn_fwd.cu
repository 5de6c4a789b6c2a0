// Forward kernel: one CTA per (work item = sequence b, q tile qt) and head h.
//
//   warp 8      TMA producer: Q tile once, then the K and V tiles of every
//               visited kv tile into two rings of kStages (3 at D=128, 4 at
//               D<=64); K runs one tile ahead and frees after QK^T, V after
//               PV, which keeps the load latency off the critical path.
//   warp 9      TMEM owner and MMA issuer (one elected lane):
//                 S[it % 3] = Q K^T             (tcgen05, SMEM x SMEM)
//                 O        += P[it % 3] V       (tcgen05, TMEM x SMEM)
//               S runs two tiles ahead of PV, so the tensor core fills one S
//               buffer while the epilogue groups work on the other two.
//   warps 0-7   epilogue, two groups of four warps that ping-pong over the kv
//               tiles: group g (warps 4g..4g+3, TMEM lanes 32(w%4)..) takes
//               the tiles it with it % 2 == g (S buffer it % 3). Per
//               tile: P' = S (1 + tanh(alpha S / 2)) (that is silu(alpha S)/N
//               up to the factor alpha / (2N), applied once to O at the
//               store), with the row's interval mask on partial tiles only
//               (full tiles run no mask arithmetic), packed to bf16 in place
//               over the first 64 columns of the buffer. While one group
//               works on tile it the other works on tile it+1, so two tiles'
//               TMEM-load / MUFU / TMEM-store latency chains overlap. At the
//               end each group stores half of O's columns (bf16, rows past
//               L_b left alone).
//
// TMEM (512 columns): S0 [0,128), S1 [128,256), S2 [256,384), O [384, 384+DP).
// Packed P of buffer b occupies columns [128b, 128b+64).
// SMEM: Q (DP/64 chunks of 128 rows x 128 B, 128-byte swizzle), K and V
// stages of the same shape.
#include "common.cuh"
#include "internal.h"

namespace hstu {

template <int DP>
struct FwdSmem {
  static constexpr int kChunks = DP / 64;
  static constexpr int kTile = kChunks * kBlock * 128;  // bytes of a 128 x DP bf16 tile
  static constexpr int kStages = DP == 128 ? 3 : 4;     // K/V ring depth
  alignas(1024) uint8_t q[kTile];
  alignas(1024) uint8_t k[kStages][kTile];
  alignas(1024) uint8_t v[kStages][kTile];
  alignas(8) uint64_t bar_q, bar_k_full[kStages], bar_k_empty[kStages], bar_v_full[kStages],
      bar_v_empty[kStages], bar_s_full[3], bar_p_full[3], bar_o_full;
  uint32_t tmem_base;
  int abort_flag;
  int n_tiles;
  int16_t tile_j[kMaxTiles];
  uint8_t tile_c[kMaxTiles];
};

template <typename S>
__device__ __forceinline__ S& smem_as(uint8_t* raw) {
  return *reinterpret_cast<S*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
}

// Warp-uniform bounded wait.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  const bool ok = mbar_wait(bar, parity, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

// P' = s (1 + tanh(alpha s / 2)) = silu(alpha s) / N / hc for 32 columns,
// packed to 16 bf16x2 words; MASKED zeroes the columns whose bit is clear.
template <bool MASKED>
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
    pk[e / 2] = pack_bf16x2(p0, p1);
  }
}

template <int DP, int NINT>
__global__ void __launch_bounds__(320, 1) hstu_fwd_kernel(const __grid_constant__ AttnParams p) {
  using Smem = FwdSmem<DP>;
  extern __shared__ uint8_t smem_raw[];
  Smem& s = smem_as<Smem>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int item = blockIdx.x / p.heads, h = blockIdx.x - item * p.heads;
  volatile int32_t* hdr = p.header;
  if (item >= hdr[kHdrNFwd] || hdr[kHdrErr] != 0) return;
  const int code = p.list[item];
  const int b = code >> 8, qt = code & 255;
  const int o0 = p.seq_offsets[b];
  const int L = p.seq_offsets[b + 1] - o0;
  const int ntiles_b = (L + kBlock - 1) / kBlock;
  const uint8_t* cls_row = p.cls + (static_cast<size_t>(b) * p.nt + qt) * p.nt;

  if (threadIdx.x == 0) {
    s.abort_flag = 0;
    mbar_init(smem_u32(&s.bar_q), 1);
    for (int i = 0; i < Smem::kStages; ++i) {
      mbar_init(smem_u32(&s.bar_k_full[i]), 1);
      mbar_init(smem_u32(&s.bar_k_empty[i]), 1);
      mbar_init(smem_u32(&s.bar_v_full[i]), 1);
      mbar_init(smem_u32(&s.bar_v_empty[i]), 1);
    }
    for (int i = 0; i < 3; ++i) {
      mbar_init(smem_u32(&s.bar_s_full[i]), 1);
      mbar_init(smem_u32(&s.bar_p_full[i]), 128);
    }
    mbar_init(smem_u32(&s.bar_o_full), 1);
    fence_mbar_init();
  }
  if (warp == 0) {  // compact list of visited kv tiles
    int n = 0;
    for (int base = 0; base < ntiles_b; base += 32) {
      const int j = base + lane;
      const uint8_t c = j < ntiles_b ? cls_row[j] : kSkip;
      const unsigned m = __ballot_sync(0xffffffffu, c != kSkip);
      if (c != kSkip) {
        const int pos = n + __popc(m & ((1u << lane) - 1u));
        s.tile_j[pos] = static_cast<int16_t>(j);
        s.tile_c[pos] = c;
      }
      n += __popc(m);
    }
    if (lane == 0) s.n_tiles = n;
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(&s.tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = s.tmem_base;
  const uint32_t tO = tbase + 384;  // O accumulator columns [384, 384 + DP)
  const int nt = s.n_tiles;
  volatile int* abort_flag = &s.abort_flag;
  const int q_row0 = o0 + qt * kBlock;
  constexpr int kTile = Smem::kTile;
  constexpr int kChunkBytes = kBlock * 128;

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (nt > 0 && elect_one_sync()) {
      // K runs one tile ahead of V: a K stage frees as soon as its QK^T has
      // completed, a V stage only after its PV, so the K load of a later
      // tile never waits behind a V slot.
      constexpr int NS = Smem::kStages;
      int k_last[NS], v_last[NS];
      for (int i = 0; i < NS; ++i) k_last[i] = v_last[i] = -1;
      mbar_expect_tx(smem_u32(&s.bar_q), kTile);
      for (int c = 0; c < Smem::kChunks; ++c)
        tma_load_3d(smem_u32(s.q + c * kChunkBytes), &p.tm_q, smem_u32(&s.bar_q), c * 64, h, q_row0);
      bool ok = true;
      for (int it = 0; ok && it <= nt; ++it) {
        if (it < nt) {  // K of tile it
          const int st = it % NS, use = it / NS;
          if (use > 0 && !mbar_wait(smem_u32(&s.bar_k_empty[st]), (use - 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t bar = smem_u32(&s.bar_k_full[st]);
          mbar_expect_tx(bar, kTile);
          const int kv_row0 = o0 + s.tile_j[it] * kBlock;
          for (int c = 0; c < Smem::kChunks; ++c)
            tma_load_3d(smem_u32(s.k[st] + c * kChunkBytes), &p.tm_k, bar, c * 64, h, kv_row0);
          k_last[st] = use;
        }
        if (it >= 1) {  // V of tile it - 1
          const int vi = it - 1, st = vi % NS, use = vi / NS;
          if (use > 0 && !mbar_wait(smem_u32(&s.bar_v_empty[st]), (use - 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t bar = smem_u32(&s.bar_v_full[st]);
          mbar_expect_tx(bar, kTile);
          const int kv_row0 = o0 + s.tile_j[vi] * kBlock;
          for (int c = 0; c < Smem::kChunks; ++c)
            tma_load_3d(smem_u32(s.v[st] + c * kChunkBytes), &p.tm_v, bar, c * 64, h, kv_row0);
          v_last[st] = use;
        }
      }
      // Never leave with a copy in flight.
      mbar_wait_drain(smem_u32(&s.bar_q), 0);
      for (int st = 0; st < NS; ++st) {
        if (k_last[st] >= 0) mbar_wait_drain(smem_u32(&s.bar_k_full[st]), k_last[st] & 1);
        if (v_last[st] >= 0) mbar_wait_drain(smem_u32(&s.bar_v_full[st]), v_last[st] & 1);
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (nt > 0 && elect_one_sync()) {
      constexpr uint32_t idesc_s = idesc_bf16(128, 128, false, false);
      constexpr uint32_t idesc_o = idesc_bf16(128, DP, false, true);
      // Descriptors are built once; each MMA only advances a start address.
      const uint64_t dq = sdesc_sw128(smem_u32(s.q), 16, 1024);
      const uint64_t dk0 = sdesc_sw128(smem_u32(s.k[0]), 16, 1024);
      const uint64_t dv0 = sdesc_sw128(smem_u32(s.v[0]), kChunkBytes, 1024);
      bool ok = mbar_wait(smem_u32(&s.bar_q), 0, abort_flag);
      tc_fence_after();
      // S runs two tiles ahead of PV: S(it) goes into buffer it % 3, whose
      // previous tile it - 3 was consumed by a PV issued before it.
      for (int it = 0; ok && it <= nt + 1; ++it) {
        if (it < nt) {
          const int kst = it % Smem::kStages, kuse = it / Smem::kStages, sb = it % 3;
          if (!mbar_wait(smem_u32(&s.bar_k_full[kst]), kuse & 1, abort_flag)) break;
          tc_fence_after();
          const uint64_t dk = sdesc_advance(dk0, kst * kTile);
          const uint32_t d_tmem = tbase + sb * 128;
#pragma unroll
          for (int kk = 0; kk < DP / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
            umma_ss(d_tmem, sdesc_advance(dq, off), sdesc_advance(dk, off), idesc_s, kk > 0);
          }
          umma_commit(smem_u32(&s.bar_s_full[sb]));
          umma_commit(smem_u32(&s.bar_k_empty[kst]));  // K stage free once QK^T is done
        }
        if (it >= 2 && it - 2 < nt) {
          const int pi = it - 2, psb = pi % 3, puse = pi / 3, pkst = pi % Smem::kStages;
          if (!mbar_wait(smem_u32(&s.bar_v_full[pkst]), (pi / Smem::kStages) & 1, abort_flag)) break;
          if (!mbar_wait(smem_u32(&s.bar_p_full[psb]), puse & 1, abort_flag)) break;
          tc_fence_after();
          const uint64_t dv = sdesc_advance(dv0, pkst * kTile);
          const uint32_t a_tmem = tbase + psb * 128;
          const uint32_t first = pi > 0 ? 1u : 0u;
          umma_ts(tO, a_tmem, dv, idesc_o, first);
#pragma unroll
          for (int kk = 1; kk < kBlock / 16; ++kk)
            umma_ts(tO, a_tmem + kk * 8, sdesc_advance(dv, kk * 16 * 128), idesc_o, 1u);
          umma_commit(smem_u32(&s.bar_v_empty[pkst]));
        }
      }
      // Arrives once every MMA issued above has completed (also on abort).
      umma_commit(smem_u32(&s.bar_o_full));
      mbar_wait_drain(smem_u32(&s.bar_o_full), 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3, half = warp >> 2;
    const int r = quarter * 32 + lane;  // q row within the tile == TMEM lane
    const int i_loc = qt * kBlock + r;
    const bool valid = i_loc < L;
    int lo[NINT], hi[NINT];
    load_row_intervals<NINT>(p.func, p.total, static_cast<int64_t>(o0) + i_loc, L, valid, lo, hi);
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const float half_alpha = 0.5f * p.alpha;
    const float out_scale = 0.5f * p.alpha * p.inv_n;  // hc = alpha / (2N)
    bool ok = true;
    // Ping-pong: warp group `half` takes the tiles it with it % 2 == half;
    // tile it lives in S buffer it % 3, so two tiles' epilogues run at the
    // same time while the tensor core fills the third buffer.
    for (int it = half; it < nt; it += 2) {
      const int sbuf = it % 3, use = it / 3;
      if (!warp_wait(smem_u32(&s.bar_s_full[sbuf]), use & 1, abort_flag)) { ok = false; break; }
      tc_fence_after();
      const int col0 = s.tile_j[it] * kBlock;
      const bool partial = s.tile_c[it] == kPartial;
      const uint32_t sb = tbase + lane_addr + sbuf * 128;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t a[32], c[32];
        tmem_ld32(sb + hf * 64, a);
        tmem_ld32(sb + hf * 64 + 32, c);
        tmem_ld_wait(a);
        tmem_ld_wait(c);
        uint32_t pa[16], pc[16];
        if (partial) {  // CTA-uniform: full tiles run no mask arithmetic
          silu_pack32<true>(a, row_mask_word<NINT>(lo, hi, col0 + hf * 64), half_alpha, pa);
          silu_pack32<true>(c, row_mask_word<NINT>(lo, hi, col0 + hf * 64 + 32), half_alpha, pc);
        } else {
          silu_pack32<false>(a, 0u, half_alpha, pa);
          silu_pack32<false>(c, 0u, half_alpha, pc);
        }
        // Packed over columns [32 hf, 32 hf + 32) of the buffer, which this
        // warp has already read: K-step kk of the PV MMA reads [8kk, 8kk+8).
        tmem_st16(sb + hf * 32, pa);
        tmem_st16(sb + hf * 32 + 16, pc);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(smem_u32(&s.bar_p_full[sbuf]));
    }
    if (ok && nt > 0) ok = warp_wait(smem_u32(&s.bar_o_full), 0, abort_flag);
    tc_fence_after();
    if (ok && !*abort_flag) {
      constexpr int kHalfCols = DP / 2;
      __nv_bfloat16* dst = p.out0 + (static_cast<int64_t>(q_row0 + r) * p.heads + h) * p.dim;
#pragma unroll
      for (int cc = 0; cc < kHalfCols / 32; ++cc) {
        const int col = half * kHalfCols + cc * 32;
        uint32_t v32[32];
        if (nt > 0) {
          tmem_ld32(tO + lane_addr + col, v32);
          tmem_ld_wait(v32);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) v32[e] = 0u;
        }
        if (valid && col < p.dim) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack_bf16x2(out_scale * __uint_as_float(v32[2 * e]),
                                out_scale * __uint_as_float(v32[2 * e + 1]));
          uint4* d4 = reinterpret_cast<uint4*>(dst + col);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            d4[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
  if (threadIdx.x == 0 && s.abort_flag) atomicOr(p.header + kHdrErr, kErrTimeout);
}

template <int DP, int NINT>
static cudaError_t launch_fwd_t(const AttnParams& p, int grid_items, cudaStream_t stream) {
  const int smem = static_cast<int>(sizeof(FwdSmem<DP>)) + 1024;
  static bool configured = false;  // attribute set once per instantiation
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(hstu_fwd_kernel<DP, NINT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const long long ctas = static_cast<long long>(grid_items) * p.heads;
  if (ctas <= 0) return cudaSuccess;
  hstu_fwd_kernel<DP, NINT><<<static_cast<unsigned>(ctas), 320, smem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_fwd(const AttnParams& p, int nint, int grid_items, cudaStream_t stream) {
  if (p.dim > 64) {
    if (nint == 1) return launch_fwd_t<128, 1>(p, grid_items, stream);
    if (nint == 2) return launch_fwd_t<128, 2>(p, grid_items, stream);
    return launch_fwd_t<128, 3>(p, grid_items, stream);
  }
  if (nint == 1) return launch_fwd_t<64, 1>(p, grid_items, stream);
  if (nint == 2) return launch_fwd_t<64, 2>(p, grid_items, stream);
  return launch_fwd_t<64, 3>(p, grid_items, stream);
}

}  // namespace hstu
