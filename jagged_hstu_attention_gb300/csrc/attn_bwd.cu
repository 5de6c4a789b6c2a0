// Backward kernel: one launch, two CTA roles taken from one longest-first
// work list (entries carry the role bit), so both run side by side.
//
// dK/dV role -- one CTA per (sequence b, kv tile kt, head h). K and V of the
// tile stay in SMEM; the Q and dO tiles of every q tile that visits kt stream
// through a 2-stage ring. Per q tile (TMEM lanes = kv rows):
//     S^T  = K Q^T,  dP^T = V dO^T                      (SMEM x SMEM)
//     P^T  = silu(alpha S^T)/N,  dS^T = dP^T * silu'(alpha S^T) * alpha/N
//            (masked on partial tiles, packed bf16 in place over S^T, dP^T)
//     dV  += P^T dO,  dK += dS^T Q                       (TMEM x SMEM)
// dK and dV accumulate in TMEM across the whole loop and are stored once:
// no atomics, fixed order, bitwise repeatable.
//
// dQ role -- one CTA per (sequence b, q tile qt, head h). Q and dO stay in
// SMEM; K and V of every visited kv tile stream. Per kv tile (lanes = q rows):
//     S = Q K^T,  dP = dO V^T;  dS = dP * silu'(alpha S) * alpha/N (packed
//     over S);  dQ += dS K.
// This recomputes S and dP once more per visible tile pair (14 D instead of
// 10 D flops per pair) in exchange for a deterministic dQ with no fp32
// workspace and no reduce-add traffic.
//
// Warps: 0-3 epilogue (one thread per TMEM lane), 4 TMA producer, 5 TMEM owner
// and MMA issuer.
#include "common.cuh"
#include "internal.h"

namespace hstu {

template <int DP>
struct BwdSmem {
  static constexpr int kChunks = DP / 64;
  static constexpr int kTile = kChunks * kBlock * 128;
  // dK/dV role: res0 = K, res1 = V, str0 = Q, str1 = dO.
  // dQ role:    res0 = Q, res1 = dO, str0 = K, str1 = V.
  alignas(1024) uint8_t res0[kTile];
  alignas(1024) uint8_t res1[kTile];
  alignas(1024) uint8_t str0[2][kTile];
  alignas(1024) uint8_t str1[2][kTile];
  alignas(8) uint64_t bar_res, bar_full[2], bar_empty[2], bar_s_full, bar_p_full, bar_acc,
      bar_func[2];
  uint32_t tmem_base;
  int abort_flag;
  int n_tiles;
  int16_t tile_idx[kMaxTiles];
  uint8_t tile_c[kMaxTiles];
  // dK/dV role: intervals of the current q tile's rows (double buffered).
  int32_t flo[2][kMaxIntervals][kBlock];
  int32_t fhi[2][kMaxIntervals][kBlock];
};

template <typename S>
__device__ __forceinline__ S& smem_as_b(uint8_t* raw) {
  return *reinterpret_cast<S*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ bool warp_wait_b(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  const bool ok = mbar_wait(bar, parity, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

// Stores 32 fp32 accumulator columns of one row as bf16.
__device__ __forceinline__ void store_row32(__nv_bfloat16* dst, const uint32_t (&a)[32]) {
  uint32_t pk[16];
#pragma unroll
  for (int e = 0; e < 16; ++e)
    pk[e] = pack_bf16x2(__uint_as_float(a[2 * e]), __uint_as_float(a[2 * e + 1]));
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int e = 0; e < 4; ++e) d4[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
}

// Writes TMEM columns [col, col + DP) of this thread's lane (or zeros) as a
// bf16 row of `dim` elements.
template <int DP>
__device__ __forceinline__ void store_acc_row(uint32_t taddr, bool have, bool valid,
                                              __nv_bfloat16* dst, int dim) {
#pragma unroll
  for (int c = 0; c < DP / 32; ++c) {
    uint32_t a[32];
    if (have) {
      tmem_ld32(taddr + c * 32, a);
      tmem_ld_wait(a);
    } else {
#pragma unroll
      for (int e = 0; e < 32; ++e) a[e] = 0u;
    }
    if (valid && c * 32 < dim) store_row32(dst + c * 32, a);
  }
}

template <int DP, int NINT>
__device__ __forceinline__ void bwd_role(const AttnParams& p, BwdSmem<DP>& s, bool dkdv, int b,
                                         int tile, int h) {
  using Smem = BwdSmem<DP>;
  constexpr int kTile = Smem::kTile;
  constexpr int kChunkBytes = kBlock * 128;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int o0 = p.seq_offsets[b];
  const int L = p.seq_offsets[b + 1] - o0;
  const int ntiles_b = (L + kBlock - 1) / kBlock;
  const size_t nt_all = static_cast<size_t>(p.nt);
  const uint8_t* cls_b = p.cls + static_cast<size_t>(b) * nt_all * nt_all;

  if (threadIdx.x == 0) {
    s.abort_flag = 0;
    mbar_init(smem_u32(&s.bar_res), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&s.bar_full[i]), 1);
      mbar_init(smem_u32(&s.bar_empty[i]), 1);
    }
    mbar_init(smem_u32(&s.bar_s_full), 1);
    mbar_init(smem_u32(&s.bar_p_full), 128);
    mbar_init(smem_u32(&s.bar_acc), 1);
    mbar_init(smem_u32(&s.bar_func[0]), 128);
    mbar_init(smem_u32(&s.bar_func[1]), 128);
    fence_mbar_init();
  }
  if (warp == 0) {
    // dK/dV: q tiles i visiting kv tile `tile` (column of the class matrix);
    // dQ: kv tiles j visited by q tile `tile` (row of the class matrix).
    int n = 0;
    for (int base = 0; base < ntiles_b; base += 32) {
      const int x = base + lane;
      uint8_t c = kSkip;
      if (x < ntiles_b) c = dkdv ? cls_b[static_cast<size_t>(x) * nt_all + tile]
                                 : cls_b[static_cast<size_t>(tile) * nt_all + x];
      const unsigned m = __ballot_sync(0xffffffffu, c != kSkip);
      if (c != kSkip) {
        const int pos = n + __popc(m & ((1u << lane) - 1u));
        s.tile_idx[pos] = static_cast<int16_t>(x);
        s.tile_c[pos] = c;
      }
      n += __popc(m);
    }
    if (lane == 0) s.n_tiles = n;
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(&s.tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = s.tmem_base;
  const int nt = s.n_tiles;
  volatile int* abort_flag = &s.abort_flag;
  const int row0 = o0 + tile * kBlock;  // rows of the resident tiles
  // TMEM columns.
  const uint32_t t_acc0 = tbase;        // dK/dV role: dV;  dQ role: dQ
  const uint32_t t_acc1 = tbase + DP;   // dK/dV role: dK
  const uint32_t t_s = dkdv ? tbase + 2 * DP : tbase + 256;
  const uint32_t t_dp = t_s + 128;
  // dQ role keeps dQ at column 256 and S/dP at 0/128.
  const uint32_t t_dq = tbase + 256;
  const uint32_t t_s_q = tbase, t_dp_q = tbase + 128;
  const uint32_t tS = dkdv ? t_s : t_s_q;
  const uint32_t tdP = dkdv ? t_dp : t_dp_q;

  const CUtensorMap* m_res0 = dkdv ? &p.tm_k : &p.tm_q;
  const CUtensorMap* m_res1 = dkdv ? &p.tm_v : &p.tm_do;
  const CUtensorMap* m_str0 = dkdv ? &p.tm_q : &p.tm_k;
  const CUtensorMap* m_str1 = dkdv ? &p.tm_do : &p.tm_v;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (nt > 0 && elect_one_sync()) {
      int last_use[2] = {-1, -1};
      const uint32_t br = smem_u32(&s.bar_res);
      mbar_expect_tx(br, 2 * kTile);
      for (int c = 0; c < Smem::kChunks; ++c) {
        tma_load_3d(smem_u32(s.res0 + c * kChunkBytes), m_res0, br, c * 64, h, row0);
        tma_load_3d(smem_u32(s.res1 + c * kChunkBytes), m_res1, br, c * 64, h, row0);
      }
      for (int it = 0; it < nt; ++it) {
        const int st = it & 1, use = it >> 1;
        if (use > 0 && !mbar_wait(smem_u32(&s.bar_empty[st]), (use - 1) & 1, abort_flag)) break;
        const int srow0 = o0 + s.tile_idx[it] * kBlock;
        const uint32_t bar = smem_u32(&s.bar_full[st]);
        mbar_expect_tx(bar, 2 * kTile);
        for (int c = 0; c < Smem::kChunks; ++c) {
          tma_load_3d(smem_u32(s.str0[st] + c * kChunkBytes), m_str0, bar, c * 64, h, srow0);
          tma_load_3d(smem_u32(s.str1[st] + c * kChunkBytes), m_str1, bar, c * 64, h, srow0);
        }
        last_use[st] = use;
      }
      mbar_wait_drain(br, 0);
      for (int st = 0; st < 2; ++st)
        if (last_use[st] >= 0) mbar_wait_drain(smem_u32(&s.bar_full[st]), last_use[st] & 1);
    }
    __syncwarp();
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (nt > 0 && elect_one_sync()) {
      constexpr uint32_t idesc_s = idesc_bf16(128, 128, false, false);
      constexpr uint32_t idesc_acc = idesc_bf16(128, DP, false, true);
      const uint32_t r0 = smem_u32(s.res0), r1 = smem_u32(s.res1);
      bool ok = mbar_wait(smem_u32(&s.bar_res), 0, abort_flag);
      tc_fence_after();
      for (int it = 0; ok && it < nt; ++it) {
        const int st = it & 1, use = it >> 1;
        if (!mbar_wait(smem_u32(&s.bar_full[st]), use & 1, abort_flag)) break;
        tc_fence_after();
        const uint32_t s0 = smem_u32(s.str0[st]), s1 = smem_u32(s.str1[st]);
        // S (or S^T) = res0 . str0^T ; dP (or dP^T) = res1 . str1^T
#pragma unroll
        for (int kk = 0; kk < DP / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
          umma_ss(tS, sdesc_sw128(r0 + off, 16, 1024), sdesc_sw128(s0 + off, 16, 1024), idesc_s,
                  kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < DP / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
          umma_ss(tdP, sdesc_sw128(r1 + off, 16, 1024), sdesc_sw128(s1 + off, 16, 1024), idesc_s,
                  kk > 0);
        }
        umma_commit(smem_u32(&s.bar_s_full));
        if (!mbar_wait(smem_u32(&s.bar_p_full), it & 1, abort_flag)) break;
        tc_fence_after();
        if (dkdv) {
          // dV += P^T dO (dO = str1, MN-major); dK += dS^T Q (Q = str0, MN-major)
#pragma unroll
          for (int kk = 0; kk < kBlock / 16; ++kk) {
            const uint32_t acc = (it > 0 || kk > 0) ? 1u : 0u;
            umma_ts(t_acc0, tS + kk * 8, sdesc_sw128(s1 + kk * 16 * 128, kChunkBytes, 1024),
                    idesc_acc, acc);
            umma_ts(t_acc1, tdP + kk * 8, sdesc_sw128(s0 + kk * 16 * 128, kChunkBytes, 1024),
                    idesc_acc, acc);
          }
        } else {
          // dQ += dS K (K = str0, MN-major)
#pragma unroll
          for (int kk = 0; kk < kBlock / 16; ++kk) {
            umma_ts(t_dq, tS + kk * 8, sdesc_sw128(s0 + kk * 16 * 128, kChunkBytes, 1024),
                    idesc_acc, (it > 0 || kk > 0) ? 1u : 0u);
          }
        }
        umma_commit(smem_u32(&s.bar_empty[st]));
      }
      umma_commit(smem_u32(&s.bar_acc));
      mbar_wait_drain(smem_u32(&s.bar_acc), 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int r = threadIdx.x;  // TMEM lane: kv row (dK/dV role) or q row (dQ role)
    const int own_loc = tile * kBlock + r;
    const bool valid = own_loc < L;
    const uint32_t lane_addr = static_cast<uint32_t>(warp * 32) << 16;
    const float alpha = p.alpha, c1 = p.alpha * p.inv_n;  // c1: alpha/N
    int lo[NINT], hi[NINT];
    if (!dkdv)
      load_row_intervals<NINT>(p.func, p.total, static_cast<int64_t>(o0) + own_loc, L, valid, lo, hi);
    bool ok = true;
    int fu = 0;  // partial tiles seen so far (dK/dV role): selects the interval buffer
    for (int it = 0; it < nt; ++it) {
      const int other = s.tile_idx[it];
      const bool partial = s.tile_c[it] == kPartial;
      const int buf = fu & 1;
      if (dkdv && partial) {
        // Intervals of the visiting q tile's rows, shared by the 128 threads.
        int flo_r[NINT], fhi_r[NINT];
        const int qi = other * kBlock + r;
        load_row_intervals<NINT>(p.func, p.total, static_cast<int64_t>(o0) + qi, L, qi < L, flo_r,
                                 fhi_r);
#pragma unroll
        for (int t = 0; t < NINT; ++t) {
          s.flo[buf][t][r] = flo_r[t];
          s.fhi[buf][t][r] = fhi_r[t];
        }
        // Bounded hand-off between the 128 epilogue threads (an mbarrier, not
        // bar.sync, so that an aborting warp cannot strand the others).
        mbar_arrive(smem_u32(&s.bar_func[buf]));
        if (!warp_wait_b(smem_u32(&s.bar_func[buf]), (fu >> 1) & 1, abort_flag)) { ok = false; break; }
        ++fu;
      }
      if (!warp_wait_b(smem_u32(&s.bar_s_full), it & 1, abort_flag)) { ok = false; break; }
      tc_fence_after();
      const int col0 = other * kBlock;  // dQ role: first kv column of the tile
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t sv[32], dv[32];
        tmem_ld32(tS + lane_addr + c * 32, sv);
        tmem_ld32(tdP + lane_addr + c * 32, dv);
        tmem_ld_wait(sv);
        tmem_ld_wait(dv);
        uint32_t mask = 0xffffffffu;
        if (partial) {
          if (dkdv) {
            mask = 0;
#pragma unroll 8
            for (int e = 0; e < 32; ++e) {
              const int qi = c * 32 + e;
              bool vis = false;
#pragma unroll
              for (int t = 0; t < NINT; ++t)
                vis |= (s.flo[buf][t][qi] <= own_loc) && (own_loc < s.fhi[buf][t][qi]);
              mask |= static_cast<uint32_t>(vis) << e;
            }
          } else {
            mask = row_mask_word<NINT>(lo, hi, col0 + c * 32);
          }
        }
        uint32_t pp[16], pd[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float g[2], pv[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const float sc = __uint_as_float(sv[e + u]);
            const float x = alpha * sc;
            const float sg = sigmoidf_fast(x);
            const float dsilu = sg * (1.0f + x * (1.0f - sg));
            const bool on = (mask >> (e + u)) & 1u;
            pv[u] = on ? c1 * sc * sg : 0.0f;
            g[u] = on ? __uint_as_float(dv[e + u]) * dsilu * c1 : 0.0f;
          }
          pp[e / 2] = pack_bf16x2(pv[0], pv[1]);
          pd[e / 2] = pack_bf16x2(g[0], g[1]);
        }
        if (dkdv) {
          tmem_st16(tS + lane_addr + c * 16, pp);
          tmem_st16(tdP + lane_addr + c * 16, pd);
        } else {
          tmem_st16(tS + lane_addr + c * 16, pd);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(smem_u32(&s.bar_p_full));
    }
    if (ok && nt > 0) ok = warp_wait_b(smem_u32(&s.bar_acc), 0, abort_flag);
    tc_fence_after();
    if (ok && !*abort_flag) {
      const int64_t row = static_cast<int64_t>(row0 + r) * p.heads + h;
      if (dkdv) {
        store_acc_row<DP>(t_acc0 + lane_addr, nt > 0, valid, p.out2 + row * p.dim, p.dim);  // dV
        store_acc_row<DP>(t_acc1 + lane_addr, nt > 0, valid, p.out1 + row * p.dim, p.dim);  // dK
      } else {
        store_acc_row<DP>(t_dq + lane_addr, nt > 0, valid, p.out0 + row * p.dim, p.dim);  // dQ
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
  if (threadIdx.x == 0 && s.abort_flag) atomicOr(p.header + kHdrErr, kErrTimeout);
}

template <int DP, int NINT>
__global__ void __launch_bounds__(192, 1) hstu_bwd_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  BwdSmem<DP>& s = smem_as_b<BwdSmem<DP>>(smem_raw);
  const int item = blockIdx.x / p.heads, h = blockIdx.x - item * p.heads;
  volatile int32_t* hdr = p.header;
  if (item >= hdr[kHdrNBwd] || hdr[kHdrErr] != 0) return;
  const int code = p.list[item];
  const bool dkdv = (code & kRoleDkdv) != 0;
  const int b = (code & ~kRoleDkdv) >> 8, tile = code & 255;
  bwd_role<DP, NINT>(p, s, dkdv, b, tile, h);
}

template <int DP, int NINT>
static cudaError_t launch_bwd_t(const AttnParams& p, int grid_items, cudaStream_t stream) {
  const int smem = static_cast<int>(sizeof(BwdSmem<DP>)) + 1024;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(hstu_bwd_kernel<DP, NINT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const long long ctas = 2LL * grid_items * p.heads;
  if (ctas <= 0) return cudaSuccess;
  hstu_bwd_kernel<DP, NINT><<<static_cast<unsigned>(ctas), 192, smem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_bwd(const AttnParams& p, int nint, int grid_items, cudaStream_t stream) {
  if (p.dim > 64) {
    if (nint == 1) return launch_bwd_t<128, 1>(p, grid_items, stream);
    if (nint == 2) return launch_bwd_t<128, 2>(p, grid_items, stream);
    return launch_bwd_t<128, 3>(p, grid_items, stream);
  }
  if (nint == 1) return launch_bwd_t<64, 1>(p, grid_items, stream);
  if (nint == 2) return launch_bwd_t<64, 2>(p, grid_items, stream);
  return launch_bwd_t<64, 3>(p, grid_items, stream);
}

}  // namespace hstu
