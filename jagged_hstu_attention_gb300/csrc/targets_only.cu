// Targets-only mode: one candidate query row per sequence against the full
// K/V of its sequence (MLCommons training PR #903, "compute the last HSTU
// layer only for the rows the loss reads"). There is one q row per (b, h), so
// the work is a matrix-vector product per sequence and head: HBM-bound, not a
// contraction worth a tensor core. It runs on CUDA cores with 16-byte
// coalesced row loads:
//
//   partial kernels -- grid (B * NC chunks of 256 keys, H); 8 warps, each warp
//                      32 keys, D/8 lanes per key (8 bf16 per lane), a key's
//                      dot products reduced with shuffles inside its lanes.
//   fold kernel     -- sums the fp32 chunk partials of each (b, h) in chunk
//                      order: a deterministic split-KV reduction.
//
// Backward writes dK/dV of every key row exactly once (rank-1 updates
// p_j dO_c and dS_j q_c; zero for keys the candidate does not see) and folds
// the dQ partials the same way as the forward folds O.
#include "common.cuh"
#include "internal.h"

namespace hstu {

constexpr int kTgtThreads = 256;

__device__ __forceinline__ void bf16x8_to_f32(const uint4 u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
__device__ __forceinline__ uint4 f32_to_bf16x8(const float (&f)[8]) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}

template <int NINT>
__device__ __forceinline__ bool in_intervals(const int (&lo)[NINT], const int (&hi)[NINT], int j) {
  bool v = false;
#pragma unroll
  for (int t = 0; t < NINT; ++t) v |= (lo[t] <= j) && (j < hi[t]);
  return v;
}

// Reduces a per-lane vector of 8 over the KPS key groups of a warp, then over
// the warps of the block, and writes the block's D-vector to `out`.
template <int D>
__device__ __forceinline__ void block_reduce_store(float (&acc)[8], float* out) {
  constexpr int LPK = D / 8;
  __shared__ float red[kTgtThreads / 32][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int off = LPK; off < 32; off <<= 1)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], off);
  if (lane < LPK)
#pragma unroll
    for (int e = 0; e < 8; ++e) red[warp][lane * 8 + e] = acc[e];
  __syncthreads();
  for (int d = threadIdx.x; d < D; d += kTgtThreads) {
    float s = 0.0f;
#pragma unroll
    for (int w = 0; w < kTgtThreads / 32; ++w) s += red[w][d];
    out[d] = s;
  }
}

template <int D, int NINT, bool BWD>
__global__ void __launch_bounds__(kTgtThreads) tgt_partial_kernel(const TgtParams p) {
  constexpr int LPK = D / 8;     // lanes per key
  constexpr int KPS = 32 / LPK;  // keys per warp step
  const int b = blockIdx.x / p.nc, chunk = blockIdx.x - b * p.nc, h = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int o0 = p.seq_offsets[b];
  const int L = p.seq_offsets[b + 1] - o0;
  if (blockIdx.x == 0 && h == 0 && threadIdx.x == 0 &&
      (p.seq_offsets[0] != 0 || static_cast<int64_t>(p.seq_offsets[p.batch]) != p.total))
    atomicOr(p.header + kHdrErr, kErrInput);  // first offset not 0 or last not total
  if (L < 0 || L > p.max_seqlen || o0 < 0 || static_cast<int64_t>(o0) + L > p.total) {
    if (chunk == 0 && h == 0 && threadIdx.x == 0) atomicOr(p.header + kHdrErr, kErrInput);
    return;
  }
  const int c0 = chunk * kTgtChunk;
  if (c0 >= L) return;
  int lo[NINT], hi[NINT];
  load_row_intervals<NINT>(p.func_c, p.batch, b, L, true, lo, hi);
  float* part = p.partial + ((static_cast<size_t>(b) * p.heads + h) * p.nc + chunk) * D;
  if (!BWD) {
    bool any = false;  // chunk-level skip: no interval meets [c0, c0 + 256)
#pragma unroll
    for (int t = 0; t < NINT; ++t) any |= (lo[t] < c0 + kTgtChunk) && (hi[t] > c0) && (hi[t] > lo[t]);
    if (!any) {
      for (int d = threadIdx.x; d < D; d += kTgtThreads) part[d] = 0.0f;
      return;
    }
  }
  const int sub = lane % LPK, kslot = lane / LPK;
  const size_t hd = static_cast<size_t>(p.heads) * D;
  const size_t qoff = (static_cast<size_t>(b) * p.heads + h) * D + sub * 8;
  float qv[8], dov[8];
  bf16x8_to_f32(*reinterpret_cast<const uint4*>(p.q_c + qoff), qv);
  if (BWD) bf16x8_to_f32(*reinterpret_cast<const uint4*>(p.do_c + qoff), dov);
  const float alpha = p.alpha, c1 = p.alpha * p.inv_n;
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.0f;

#pragma unroll 4
  for (int step = 0; step < 32 / KPS; ++step) {
    const int key = c0 + warp * 32 + step * KPS + kslot;
    const bool in_range = key < L;
    const bool vis = in_range && in_intervals<NINT>(lo, hi, key);
    const size_t roff = (static_cast<size_t>(o0) + key) * hd + static_cast<size_t>(h) * D + sub * 8;
    float kf[8], vf[8];
    uint4 ku = make_uint4(0, 0, 0, 0), vu = make_uint4(0, 0, 0, 0);
    if (in_range) {
      ku = __ldg(reinterpret_cast<const uint4*>(p.k + roff));
      vu = __ldg(reinterpret_cast<const uint4*>(p.v + roff));
    }
    bf16x8_to_f32(ku, kf);
    bf16x8_to_f32(vu, vf);
    float dot = 0.0f, dot2 = 0.0f;
#pragma unroll
    for (int e = 0; e < 8; ++e) dot = fmaf(qv[e], kf[e], dot);
    if (BWD)
#pragma unroll
      for (int e = 0; e < 8; ++e) dot2 = fmaf(dov[e], vf[e], dot2);
#pragma unroll
    for (int off = LPK / 2; off > 0; off >>= 1) {
      dot += __shfl_xor_sync(0xffffffffu, dot, off);
      if (BWD) dot2 += __shfl_xor_sync(0xffffffffu, dot2, off);
    }
    const float x = alpha * dot;
    const float sg = sigmoidf_fast(x);
    if (!BWD) {
      const float pv = vis ? c1 * dot * sg : 0.0f;
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = fmaf(pv, vf[e], acc[e]);
    } else {
      const float pv = vis ? c1 * dot * sg : 0.0f;
      const float ds = vis ? dot2 * sg * (1.0f + x * (1.0f - sg)) * c1 : 0.0f;
      if (in_range) {
        float dvv[8], dkv[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          dvv[e] = pv * dov[e];
          dkv[e] = ds * qv[e];
        }
        *reinterpret_cast<uint4*>(p.dv + roff) = f32_to_bf16x8(dvv);
        *reinterpret_cast<uint4*>(p.dk + roff) = f32_to_bf16x8(dkv);
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = fmaf(ds, kf[e], acc[e]);
    }
  }
  block_reduce_store<D>(acc, part);
}

template <int D>
__global__ void __launch_bounds__(128) tgt_fold_kernel(const TgtParams p, __nv_bfloat16* out) {
  const int bh = blockIdx.x;
  const int b = bh / p.heads;
  if (p.header[kHdrErr] != 0) return;
  int L = p.seq_offsets[b + 1] - p.seq_offsets[b];
  L = min(max(L, 0), p.max_seqlen);
  const int nchunks = (L + kTgtChunk - 1) / kTgtChunk;
  const float* part = p.partial + static_cast<size_t>(bh) * p.nc * D;
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float s = 0.0f;
    for (int c = 0; c < nchunks; ++c) s += part[static_cast<size_t>(c) * D + d];
    out[static_cast<size_t>(bh) * D + d] = __float2bfloat16_rn(s);
  }
}

template <int D, bool BWD>
static cudaError_t launch_tgt_t(const TgtParams& p, cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>(p.batch) * p.nc, p.heads);
  const int nint = (p.nfunc + 1) / 2;
  switch (nint) {
    case 1: tgt_partial_kernel<D, 1, BWD><<<grid, kTgtThreads, 0, stream>>>(p); break;
    case 2: tgt_partial_kernel<D, 2, BWD><<<grid, kTgtThreads, 0, stream>>>(p); break;
    case 3: tgt_partial_kernel<D, 3, BWD><<<grid, kTgtThreads, 0, stream>>>(p); break;
    case 4: tgt_partial_kernel<D, 4, BWD><<<grid, kTgtThreads, 0, stream>>>(p); break;
    default: tgt_partial_kernel<D, 5, BWD><<<grid, kTgtThreads, 0, stream>>>(p); break;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  tgt_fold_kernel<D><<<p.batch * p.heads, 128, 0, stream>>>(p, BWD ? p.dq_c : p.o_c);
  return cudaGetLastError();
}

template <bool BWD>
static cudaError_t launch_tgt(const TgtParams& p, cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(p.header, 0, kHdrWords * 4, stream);
  if (e != cudaSuccess) return e;
  if (p.dim == 128) return launch_tgt_t<128, BWD>(p, stream);
  if (p.dim == 64) return launch_tgt_t<64, BWD>(p, stream);
  return launch_tgt_t<32, BWD>(p, stream);
}

cudaError_t launch_targets_fwd(const TgtParams& p, cudaStream_t stream) {
  return launch_tgt<false>(p, stream);
}
cudaError_t launch_targets_bwd(const TgtParams& p, cudaStream_t stream) {
  return launch_tgt<true>(p, stream);
}

}  // namespace hstu
