// Targets-only mode: candidate query rows against the full K/V of their
// sequence (MLCommons training PR #903, "compute the last HSTU layer only for
// the rows the loss reads"). There is one q row per (candidate, head), so the
// work is a matrix-vector product per candidate and head: HBM-bound, not a
// contraction worth a tensor core. It runs on CUDA cores with 16-byte
// coalesced row loads:
//
//   partial kernels -- grid (C * NC chunks of 256 keys, H) for C candidates;
//                      8 warps, each warp 32 keys, DM/8 lanes per key (8
//                      elements per lane, DM the wider of D_qk and D_v; lanes
//                      past the narrower width hold zeros), a key's dot
//                      products reduced with shuffles inside its lanes.
//   fold kernel     -- sums the fp32 chunk partials of each (candidate, h) in
//                      chunk order: a deterministic split-KV reduction.
//
// One candidate per sequence (the page's case; cand_offsets absent, candidate
// b belongs to sequence b): the backward partial kernel also writes dK/dV of
// every key row of its chunk exactly once (rank-1 updates p_j dO_c and
// dS_j q_c; zero for keys the candidate does not see).
//
// Several candidates per sequence (the page's "not exactly one target per
// sequence" batches; candidates cand_offsets[b] .. cand_offsets[b+1] belong
// to sequence b): dK_j and dV_j sum over the sequence's candidates, so a
// separate kernel, grid (B * NC, H), takes each key of a chunk through the
// sequence's candidates in order and writes its rows once (deterministic, no
// atomics); the partial kernel then only folds dQ.
#include "common.cuh"
#include "internal.h"

namespace hstu {

constexpr int kTgtThreads = 256;
// What a partial kernel computes.
constexpr int kTgtFwd = 0;       // partial O rows
constexpr int kTgtBwdFused = 1;  // one candidate per sequence: partial dQ rows and the chunk's dK/dV rows
constexpr int kTgtBwdDq = 2;     // several candidates per sequence: partial dQ rows only

// Sequence of candidate c: without cand_offsets c itself, else the largest b
// with cand_offsets[b] <= c (callers check that c < cand_offsets[b + 1]).
__device__ __forceinline__ int cand_seq(const TgtParams& p, int c) {
  if (!p.cand_offsets) return c;
  int lo = 0, hi = p.batch;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (p.cand_offsets[mid] <= c) lo = mid;
    else hi = mid;
  }
  return lo;
}

// Checks shared by the kernels that read sequence b: its offsets (every
// length in [0, max_seqlen], inside [0, total]); block (0, 0) also checks the
// first and last offsets of seq_offsets and cand_offsets. On a bad value the
// error word gets kErrInput and the caller returns.
__device__ __forceinline__ bool tgt_sequence_ok(const TgtParams& p, int b, bool reporter, int& o0, int& L) {
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
    bool bad = p.seq_offsets[0] != 0 || static_cast<int64_t>(p.seq_offsets[p.batch]) != p.total;
    if (p.cand_offsets) bad = bad || p.cand_offsets[0] != 0 || p.cand_offsets[p.batch] != p.num_cand;
    if (bad) atomicOr(p.header + kHdrErr, kErrInput);
  }
  o0 = p.seq_offsets[b];
  L = p.seq_offsets[b + 1] - o0;
  if (L < 0 || L > p.max_seqlen || o0 < 0 || static_cast<int64_t>(o0) + L > p.total) {
    if (reporter && threadIdx.x == 0) atomicOr(p.header + kHdrErr, kErrInput);
    return false;
  }
  return true;
}

template <typename T>
__device__ __forceinline__ void x8_to_f32(const uint4 u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = Elem<T>::lo(w[i]);
    f[2 * i + 1] = Elem<T>::hi(w[i]);
  }
}
template <typename T>
__device__ __forceinline__ uint4 f32_to_x8(const float (&f)[8]) {
  return make_uint4(Elem<T>::pack2(f[0], f[1]), Elem<T>::pack2(f[2], f[3]), Elem<T>::pack2(f[4], f[5]),
                    Elem<T>::pack2(f[6], f[7]));
}

__device__ __forceinline__ bool in_intervals(const int (&lo)[kMaxIntervals], const int (&hi)[kMaxIntervals],
                                             int nint, int j) {
  bool v = false;
#pragma unroll
  for (int t = 0; t < kMaxIntervals; ++t) v |= (t < nint) && (lo[t] <= j) && (j < hi[t]);
  return v;
}

// Reduces a per-lane vector of 8 over the key groups of a warp (LPK lanes
// per key), then over the warps of the block, and writes the block's
// DOUT-vector (DOUT <= 8 LPK) to `out`.
template <int LPK, int DOUT>
__device__ __forceinline__ void block_reduce_store(float (&acc)[8], float* out) {
  __shared__ float red[kTgtThreads / 32][8 * LPK];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int off = LPK; off < 32; off <<= 1)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], off);
  if (lane < LPK)
#pragma unroll
    for (int e = 0; e < 8; ++e) red[warp][lane * 8 + e] = acc[e];
  __syncthreads();
  for (int d = threadIdx.x; d < DOUT; d += kTgtThreads) {
    float s = 0.0f;
#pragma unroll
    for (int w = 0; w < kTgtThreads / 32; ++w) s += red[w][d];
    out[d] = s;
  }
}

template <typename T, int DQ, int DV, int MODE>
__global__ void __launch_bounds__(kTgtThreads, 5) tgt_partial_kernel(const TgtParams p) {
  constexpr bool BWD = MODE != kTgtFwd;
  constexpr int DM = DQ > DV ? DQ : DV;
  constexpr int LPK = DM / 8;    // lanes per key
  constexpr int KPS = 32 / LPK;  // keys per warp step
  constexpr int DOUT = BWD ? DQ : DV;  // partial rows: dQ (backward) or O (forward)
  const int cand = blockIdx.x / p.nc, chunk = blockIdx.x - cand * p.nc, h = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = cand_seq(p, cand);
  if (p.cand_offsets && !(p.cand_offsets[b] <= cand && cand < p.cand_offsets[b + 1])) {
    if (chunk == 0 && h == 0 && threadIdx.x == 0) atomicOr(p.header + kHdrErr, kErrInput);
    return;  // cand_offsets out of order
  }
  int o0, L;
  if (!tgt_sequence_ok(p, b, chunk == 0 && h == 0, o0, L)) return;
  const int c0 = chunk * kTgtChunk;
  if (c0 >= L) return;
  const int nint = (p.nfunc + 1) / 2;
  int lo[kMaxIntervals], hi[kMaxIntervals];
  load_row_intervals<kMaxIntervals>(p.func_c, p.num_cand, cand, L, true, lo, hi, (1u << nint) - 1u);
  float* part = p.partial + ((static_cast<size_t>(cand) * p.heads + h) * p.nc + chunk) * DM;
  if (!BWD) {
    bool any = false;  // chunk-level skip: no interval meets [c0, c0 + 256)
#pragma unroll
    for (int t = 0; t < kMaxIntervals; ++t) any |= (lo[t] < c0 + kTgtChunk) && (hi[t] > c0) && (hi[t] > lo[t]);
    if (!any) {
      for (int d = threadIdx.x; d < DOUT; d += kTgtThreads) part[d] = 0.0f;
      return;
    }
  }
  const int sub = lane % LPK, kslot = lane / LPK;
  // This lane's 8 columns exist in the q/k rows (DQ wide) and the v/dO rows (DV wide)?
  const bool has_q = sub * 8 < DQ, has_v = sub * 8 < DV;
  const size_t hdq = static_cast<size_t>(p.heads) * DQ, hdv = static_cast<size_t>(p.heads) * DV;
  const size_t bh = static_cast<size_t>(cand) * p.heads + h;
  const T* qc = static_cast<const T*>(p.q_c);
  const T* kp = static_cast<const T*>(p.k);
  const T* vp = static_cast<const T*>(p.v);
  float qv[8], dov[8];
  const uint4 zero4 = make_uint4(0, 0, 0, 0);
  x8_to_f32<T>(has_q ? *reinterpret_cast<const uint4*>(qc + bh * DQ + sub * 8) : zero4, qv);
  if (BWD)
    x8_to_f32<T>(has_v ? *reinterpret_cast<const uint4*>(static_cast<const T*>(p.do_c) + bh * DV + sub * 8) : zero4,
                 dov);
  const float alpha = p.alpha, c1 = p.alpha * p.inv_n;
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.0f;

#pragma unroll 4
  for (int step = 0; step < 32 / KPS; ++step) {
    const int key = c0 + warp * 32 + step * KPS + kslot;
    const bool in_range = key < L;
    const bool vis = in_range && in_intervals(lo, hi, nint, key);
    const size_t krow = static_cast<size_t>(o0) + key;
    const size_t koff = krow * hdq + static_cast<size_t>(h) * DQ + sub * 8;
    const size_t voff = krow * hdv + static_cast<size_t>(h) * DV + sub * 8;
    float kf[8], vf[8];
    uint4 ku = zero4, vu = zero4;
    if (in_range && has_q) ku = __ldg(reinterpret_cast<const uint4*>(kp + koff));
    if (in_range && has_v) vu = __ldg(reinterpret_cast<const uint4*>(vp + voff));
    x8_to_f32<T>(ku, kf);
    x8_to_f32<T>(vu, vf);
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
      if (MODE == kTgtBwdFused && in_range) {
        float dvv[8], dkv[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          dvv[e] = pv * dov[e];
          dkv[e] = ds * qv[e];
        }
        if (has_v) *reinterpret_cast<uint4*>(static_cast<T*>(p.dv) + voff) = f32_to_x8<T>(dvv);
        if (has_q) *reinterpret_cast<uint4*>(static_cast<T*>(p.dk) + koff) = f32_to_x8<T>(dkv);
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = fmaf(ds, kf[e], acc[e]);
    }
  }
  block_reduce_store<LPK, DOUT>(acc, part);
}

// dK/dV rows of one chunk of keys of sequence b when a sequence may have
// several candidates: each key goes through the sequence's candidates in
// order (fixed order, no atomics) and its rows are written once; keys no
// candidate sees get zeros.
template <typename T, int DQ, int DV>
__global__ void __launch_bounds__(kTgtThreads, 3) tgt_dkdv_kernel(const TgtParams p) {
  constexpr int DM = DQ > DV ? DQ : DV;
  constexpr int LPK = DM / 8;
  constexpr int KPS = 32 / LPK;
  const int b = blockIdx.x / p.nc, chunk = blockIdx.x - b * p.nc, h = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int o0, L;
  if (!tgt_sequence_ok(p, b, chunk == 0 && h == 0, o0, L)) return;
  const int k0 = chunk * kTgtChunk;
  if (k0 >= L) return;
  const int cb = p.cand_offsets[b], ce = p.cand_offsets[b + 1];
  if (cb < 0 || ce < cb || ce > p.num_cand) {
    if (chunk == 0 && h == 0 && threadIdx.x == 0) atomicOr(p.header + kHdrErr, kErrInput);
    return;
  }
  const int nint = (p.nfunc + 1) / 2;
  const int sub = lane % LPK, kslot = lane / LPK;
  const bool has_q = sub * 8 < DQ, has_v = sub * 8 < DV;
  const size_t hdq = static_cast<size_t>(p.heads) * DQ, hdv = static_cast<size_t>(p.heads) * DV;
  const T* qc = static_cast<const T*>(p.q_c);
  const T* dc = static_cast<const T*>(p.do_c);
  const T* kp = static_cast<const T*>(p.k);
  const T* vp = static_cast<const T*>(p.v);
  const uint4 zero4 = make_uint4(0, 0, 0, 0);
  const float alpha = p.alpha, c1 = p.alpha * p.inv_n;
  for (int step = 0; step < 32 / KPS; ++step) {
    const int key = k0 + warp * 32 + step * KPS + kslot;
    const bool in_range = key < L;
    const size_t krow = static_cast<size_t>(o0) + key;
    const size_t koff = krow * hdq + static_cast<size_t>(h) * DQ + sub * 8;
    const size_t voff = krow * hdv + static_cast<size_t>(h) * DV + sub * 8;
    float kf[8], vf[8], dk[8], dv[8];
    x8_to_f32<T>(in_range && has_q ? __ldg(reinterpret_cast<const uint4*>(kp + koff)) : zero4, kf);
    x8_to_f32<T>(in_range && has_v ? __ldg(reinterpret_cast<const uint4*>(vp + voff)) : zero4, vf);
#pragma unroll
    for (int e = 0; e < 8; ++e) dk[e] = dv[e] = 0.0f;
    for (int c = cb; c < ce; ++c) {
      int lo[kMaxIntervals], hi[kMaxIntervals];
      load_row_intervals<kMaxIntervals>(p.func_c, p.num_cand, c, L, true, lo, hi, (1u << nint) - 1u);
      const bool vis = in_range && in_intervals(lo, hi, nint, key);
      const size_t bh = static_cast<size_t>(c) * p.heads + h;
      float qv[8], dov[8];
      x8_to_f32<T>(has_q ? __ldg(reinterpret_cast<const uint4*>(qc + bh * DQ + sub * 8)) : zero4, qv);
      x8_to_f32<T>(has_v ? __ldg(reinterpret_cast<const uint4*>(dc + bh * DV + sub * 8)) : zero4, dov);
      float dot = 0.0f, dot2 = 0.0f;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        dot = fmaf(qv[e], kf[e], dot);
        dot2 = fmaf(dov[e], vf[e], dot2);
      }
#pragma unroll
      for (int off = LPK / 2; off > 0; off >>= 1) {
        dot += __shfl_xor_sync(0xffffffffu, dot, off);
        dot2 += __shfl_xor_sync(0xffffffffu, dot2, off);
      }
      const float x = alpha * dot;
      const float sg = sigmoidf_fast(x);
      const float pv = vis ? c1 * dot * sg : 0.0f;
      const float ds = vis ? dot2 * sg * (1.0f + x * (1.0f - sg)) * c1 : 0.0f;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        dv[e] = fmaf(pv, dov[e], dv[e]);
        dk[e] = fmaf(ds, qv[e], dk[e]);
      }
    }
    if (in_range) {
      if (has_v) *reinterpret_cast<uint4*>(static_cast<T*>(p.dv) + voff) = f32_to_x8<T>(dv);
      if (has_q) *reinterpret_cast<uint4*>(static_cast<T*>(p.dk) + koff) = f32_to_x8<T>(dk);
    }
  }
}

// Sums the chunk partials of each (candidate, h) in chunk order into a
// DOUT-wide output row (partials are DM apart).
template <typename T, int DOUT, int DM>
__global__ void __launch_bounds__(128) tgt_fold_kernel(const TgtParams p, T* out) {
  const int bh = blockIdx.x;
  const int b = cand_seq(p, bh / p.heads);
  if (p.header[kHdrErr] != 0) return;
  int L = p.seq_offsets[b + 1] - p.seq_offsets[b];
  L = min(max(L, 0), p.max_seqlen);
  const int nchunks = (L + kTgtChunk - 1) / kTgtChunk;
  const float* part = p.partial + static_cast<size_t>(bh) * p.nc * DM;
  for (int d = threadIdx.x; d < DOUT; d += blockDim.x) {
    float s = 0.0f;
    for (int c = 0; c < nchunks; ++c) s += part[static_cast<size_t>(c) * DM + d];
    uint32_t w = Elem<T>::pack2(s, 0.0f);
    out[static_cast<size_t>(bh) * DOUT + d] = *reinterpret_cast<T*>(&w);
  }
}

template <typename T, int DQ, int DV, bool BWD>
static cudaError_t launch_tgt_t(const TgtParams& p, cudaStream_t stream) {
  constexpr int DM = DQ > DV ? DQ : DV;
  const long long blocks = static_cast<long long>(p.num_cand) * p.nc;
  if (blocks > 0x7fffffffLL || static_cast<long long>(p.batch) * p.nc > 0x7fffffffLL ||
      static_cast<long long>(p.num_cand) * p.heads > 0x7fffffffLL || p.heads > 65535)
    return cudaErrorInvalidConfiguration;
  const bool multi = p.cand_offsets != nullptr;
  if (BWD && multi) {
    const dim3 gk(static_cast<unsigned>(p.batch) * p.nc, p.heads);
    tgt_dkdv_kernel<T, DQ, DV><<<gk, kTgtThreads, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (blocks == 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>(blocks), p.heads);
  if (!BWD) tgt_partial_kernel<T, DQ, DV, kTgtFwd><<<grid, kTgtThreads, 0, stream>>>(p);
  else if (multi) tgt_partial_kernel<T, DQ, DV, kTgtBwdDq><<<grid, kTgtThreads, 0, stream>>>(p);
  else tgt_partial_kernel<T, DQ, DV, kTgtBwdFused><<<grid, kTgtThreads, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  tgt_fold_kernel<T, BWD ? DQ : DV, DM><<<static_cast<unsigned>(p.num_cand) * p.heads, 128, 0, stream>>>(
      p, static_cast<T*>(BWD ? p.dq_c : p.o_c));
  return cudaGetLastError();
}

template <typename T, int DQ, bool BWD>
static cudaError_t launch_tgt_dq(const TgtParams& p, cudaStream_t stream) {
  if (p.dim_v == 128) return launch_tgt_t<T, DQ, 128, BWD>(p, stream);
  if (p.dim_v == 64) return launch_tgt_t<T, DQ, 64, BWD>(p, stream);
  return launch_tgt_t<T, DQ, 32, BWD>(p, stream);
}

template <typename T, bool BWD>
static cudaError_t launch_tgt_typed(const TgtParams& p, cudaStream_t stream) {
  if (p.dim == 128) return launch_tgt_dq<T, 128, BWD>(p, stream);
  if (p.dim == 64) return launch_tgt_dq<T, 64, BWD>(p, stream);
  return launch_tgt_dq<T, 32, BWD>(p, stream);
}

template <bool BWD>
static cudaError_t launch_tgt(const TgtParams& p, int dtype, cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(p.header, 0, kHdrWords * 4, stream);
  if (e != cudaSuccess) return e;
  return dtype == kDtypeF16 ? launch_tgt_typed<__half, BWD>(p, stream)
                            : launch_tgt_typed<__nv_bfloat16, BWD>(p, stream);
}

cudaError_t launch_targets_fwd(const TgtParams& p, int dtype, cudaStream_t stream) {
  return launch_tgt<false>(p, dtype, stream);
}
cudaError_t launch_targets_bwd(const TgtParams& p, int dtype, cudaStream_t stream) {
  return launch_tgt<true>(p, dtype, stream);
}

}  // namespace hstu
