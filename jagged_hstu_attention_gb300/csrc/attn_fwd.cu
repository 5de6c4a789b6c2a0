// Forward kernel: one CTA per (work item = sequence b, q tile qt) and head h.
//
//   warp 8      TMA producer: Q tile once, then K/V tiles of every visited kv
//               tile into a ring of kStages (3 at D=128, 4 at D<=64).
//   warp 9      TMEM owner and MMA issuer (one elected lane):
//                 S[it % 2] = Q K^T             (tcgen05, SMEM x SMEM)
//                 O        += P[it % 2] V       (tcgen05, TMEM x SMEM)
//               S for tile it+1 is issued before P of tile it is consumed, so
//               the tensor core works while the epilogue computes P.
//   warps 0-7   epilogue. Warp w reads TMEM lanes 32(w%4).. (q rows) and the
//               column half w/4 of S: P = silu(alpha S) / N with the row's
//               interval mask on partial tiles only, packed to bf16 in place
//               over the first 32 columns of its own half (so the two halves
//               never touch each other's columns); at the end O -> bf16 ->
//               global, rows past L_b left alone. Two warps per SM
//               sub-partition hide the MUFU and TMEM latencies.
//
// TMEM (512 columns): S0 [0,128), S1 [128,256), O [256, 256+DP). Packed P of
// buffer b: K-steps 0-3 at columns [128b, 128b+32), 4-7 at [128b+64, 128b+96).
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
  alignas(8) uint64_t bar_q, bar_kv_full[kStages], bar_kv_empty[kStages], bar_s_full[2],
      bar_p_full[2], bar_o_full;
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

// P = silu(alpha s) / N for 32 columns, masked by bit k of `mask`, packed to
// 16 bf16x2 words.
__device__ __forceinline__ void silu_pack32(const uint32_t (&s)[32], uint32_t mask,
                                            const SiluConsts& kc, uint32_t (&pk)[16]) {
#pragma unroll
  for (int e = 0; e < 32; e += 2) {
    float p0 = silu_p(__uint_as_float(s[e]), kc);
    float p1 = silu_p(__uint_as_float(s[e + 1]), kc);
    p0 = ((mask >> e) & 1u) ? p0 : 0.0f;
    p1 = ((mask >> (e + 1)) & 1u) ? p1 : 0.0f;
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
      mbar_init(smem_u32(&s.bar_kv_full[i]), 1);
      mbar_init(smem_u32(&s.bar_kv_empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&s.bar_s_full[i]), 1);
      mbar_init(smem_u32(&s.bar_p_full[i]), 256);
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
  const int nt = s.n_tiles;
  volatile int* abort_flag = &s.abort_flag;
  const int q_row0 = o0 + qt * kBlock;
  constexpr int kTile = Smem::kTile;
  constexpr int kChunkBytes = kBlock * 128;

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (nt > 0 && elect_one_sync()) {
      int last_use[Smem::kStages];
      for (int i = 0; i < Smem::kStages; ++i) last_use[i] = -1;
      mbar_expect_tx(smem_u32(&s.bar_q), kTile);
      for (int c = 0; c < Smem::kChunks; ++c)
        tma_load_3d(smem_u32(s.q + c * kChunkBytes), &p.tm_q, smem_u32(&s.bar_q), c * 64, h, q_row0);
      for (int it = 0; it < nt; ++it) {
        const int st = it % Smem::kStages, use = it / Smem::kStages;
        if (use > 0 && !mbar_wait(smem_u32(&s.bar_kv_empty[st]), (use - 1) & 1, abort_flag)) break;
        const int kv_row0 = o0 + s.tile_j[it] * kBlock;
        const uint32_t bar = smem_u32(&s.bar_kv_full[st]);
        mbar_expect_tx(bar, 2 * kTile);
        for (int c = 0; c < Smem::kChunks; ++c) {
          tma_load_3d(smem_u32(s.k[st] + c * kChunkBytes), &p.tm_k, bar, c * 64, h, kv_row0);
          tma_load_3d(smem_u32(s.v[st] + c * kChunkBytes), &p.tm_v, bar, c * 64, h, kv_row0);
        }
        last_use[st] = use;
      }
      // Never leave with a copy in flight.
      mbar_wait_drain(smem_u32(&s.bar_q), 0);
      for (int st = 0; st < Smem::kStages; ++st)
        if (last_use[st] >= 0) mbar_wait_drain(smem_u32(&s.bar_kv_full[st]), last_use[st] & 1);
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (nt > 0 && elect_one_sync()) {
      constexpr uint32_t idesc_s = idesc_bf16(128, 128, false, false);
      constexpr uint32_t idesc_o = idesc_bf16(128, DP, false, true);
      const uint32_t q_base = smem_u32(s.q);
      bool ok = mbar_wait(smem_u32(&s.bar_q), 0, abort_flag);
      tc_fence_after();
      for (int it = 0; ok && it <= nt; ++it) {
        if (it < nt) {
          const int kst = it % Smem::kStages, kuse = it / Smem::kStages, sb = it & 1;
          if (!mbar_wait(smem_u32(&s.bar_kv_full[kst]), kuse & 1, abort_flag)) break;
          tc_fence_after();
          const uint32_t k_base = smem_u32(s.k[kst]);
#pragma unroll
          for (int kk = 0; kk < DP / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
            umma_ss(tbase + sb * 128, sdesc_sw128(q_base + off, 16, 1024),
                    sdesc_sw128(k_base + off, 16, 1024), idesc_s, kk > 0);
          }
          umma_commit(smem_u32(&s.bar_s_full[sb]));
        }
        if (it >= 1) {
          const int pi = it - 1, psb = pi & 1, puse = pi >> 1, pkst = pi % Smem::kStages;
          if (!mbar_wait(smem_u32(&s.bar_p_full[psb]), puse & 1, abort_flag)) break;
          tc_fence_after();
          const uint32_t v_base = smem_u32(s.v[pkst]);
#pragma unroll
          for (int kk = 0; kk < kBlock / 16; ++kk) {
            umma_ts(tbase + 256, tbase + psb * 128 + (kk >> 2) * 64 + (kk & 3) * 8,
                    sdesc_sw128(v_base + kk * 16 * 128, kChunkBytes, 1024), idesc_o,
                    (pi > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(smem_u32(&s.bar_kv_empty[pkst]));
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
    const SiluConsts kc(p.alpha, p.inv_n);
    const int hc = half * 64;  // first S column of this warp's half
    bool ok = true;
    for (int it = 0; it < nt; ++it) {
      const int st = it & 1, use = it >> 1;
      if (!warp_wait(smem_u32(&s.bar_s_full[st]), use & 1, abort_flag)) { ok = false; break; }
      tc_fence_after();
      const int col0 = s.tile_j[it] * kBlock + hc;
      const bool partial = s.tile_c[it] == kPartial;
      const uint32_t sb = tbase + lane_addr + st * 128 + hc;
      uint32_t a[32], c[32];
      tmem_ld32(sb, a);
      tmem_ld32(sb + 32, c);
      tmem_ld_wait(a);
      tmem_ld_wait(c);
      uint32_t m0 = 0xffffffffu, m1 = 0xffffffffu;
      if (partial) {
        m0 = row_mask_word<NINT>(lo, hi, col0);
        m1 = row_mask_word<NINT>(lo, hi, col0 + 32);
      }
      uint32_t pa[16], pc[16];
      silu_pack32(a, m0, kc, pa);
      silu_pack32(c, m1, kc, pc);
      tmem_st16(sb, pa);
      tmem_st16(sb + 16, pc);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(smem_u32(&s.bar_p_full[st]));
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
          tmem_ld32(tbase + lane_addr + 256 + col, v32);
          tmem_ld_wait(v32);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) v32[e] = 0u;
        }
        if (valid && col < p.dim) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack_bf16x2(__uint_as_float(v32[2 * e]), __uint_as_float(v32[2 * e + 1]));
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
