// Candidate-row projection of the targets-only layer (MLCommons training PR
// #903, Summary: the last layer computes U and Q for the candidate rows
// alone; K and V stay full length). The projection of a row is the layer's
// pointwise-SiLU input projection, y = silu(x W^T + b), W laid out (out
// features, in features); here it runs on a list of rows only.
//
//   forward   gather the listed rows of x (one small copy kernel), then one
//             tcgen05 GEMM Z = X_c W^T with the bias and SiLU fused into its
//             epilogue (y, and optionally z for the backward);
//   backward  G = dY * silu'(Z) and the bias gradient's column partials (one
//             elementwise kernel, a fixed-order fold), then two tcgen05 GEMMs:
//             dX_c = G W and dW = G^T X_c.
//
// The GEMM: C[M x N] = A[M x K] B[N x K]^T with fp32 accumulation in TMEM. A
// and B come from row-major 2-D tensors; an operand is K-major when K runs
// along the tensor's rows (A = X_c, A = G, B = W in the forward) and
// MN-major when K runs down its columns (B = W in dX_c; A = G and B = X_c in
// dW). Persistent: one CTA per SM takes output tiles of 128 x 256 in turn,
// N fastest: the CTAs running together cover every N tile of a few row
// blocks, so the long A operand (X_c, G) comes from HBM once and W, which is
// small, stays in L2 (with M fastest, A was read once per N tile); 64-deep K
// blocks flow through a 4-stage TMA ring (48 KB a stage, 128-byte swizzle)
// that runs on across tiles; one elected thread issues M=128, N=256, K=16
// MMAs into one of two 256-column TMEM accumulators, so that four epilogue
// warps read one tile out (a row per thread) while the next accumulates; the
// 16-bit results leave through each warp's shared-memory staging buffer as
// TMA stores of 32 rows x 64 columns.
// dW, whose K is the number of rows, splits K over up to eight tiles per
// output tile; their fp32 partial tiles are summed in split order
// (deterministic) by a fold kernel.
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "../../include/hstu_attn.h"
#include "common.cuh"

namespace hstu {

namespace {

constexpr int kGemmBM = 128, kGemmBN = 256, kGemmBK = 64, kGemmStages = 4;
constexpr int kMaxKSplits = 8;
// The SiLU gradient splits the rows into at most kGradChunks chunks of at
// least kGradMinRows rows (one block each); a chunk's column sums are the
// bias gradient's partials, folded in chunk order.
constexpr int kGradChunks = 1216, kGradMinRows = 64, kGradThreads = 256;
inline int grad_chunks(int64_t n) {
  const int64_t c = (n + kGradMinRows - 1) / kGradMinRows;
  return static_cast<int>(c < kGradChunks ? c : kGradChunks);
}
constexpr int kGemmThreads = 192;  // warps 0-3 epilogue, 4 TMA producer, 5 MMA issuer

// Epilogues.
constexpr int kEpiStore = 0;     // out = acc
constexpr int kEpiBiasSilu = 1;  // z = acc + bias; out = silu(z); out2 = z (optional)
constexpr int kEpiPartial = 2;   // partial[split] = acc in fp32 (split K)

struct GemmParams {
  CUtensorMap tm_a, tm_b;
  CUtensorMap tm_out, tm_out2;  // 16-bit outputs (boxes of 64 columns x 32 rows), stored by TMA
  void* out;
  void* out2;
  const void* bias;
  int32_t* err;  // error word (nullable): kErrTimeout on a timed-out wait
  float* partial;  // kEpiPartial: (k_splits, M, N) fp32
  int32_t M, N, K, ldo, k_splits;
};

struct GemmSmem {
  alignas(1024) uint8_t a[kGemmStages][kGemmBM * kGemmBK * 2];  // 16 KB a stage
  alignas(1024) uint8_t b[kGemmStages][kGemmBN * kGemmBK * 2];  // 32 KB a stage
  // Output staging of each epilogue warp: its 32 rows x 64 columns of out
  // and of out2, 128-byte rows in the 128-byte swizzle the TMA store reads.
  alignas(1024) uint8_t stage_out[4][32 * 128];
  alignas(1024) uint8_t stage_out2[4][32 * 128];
  alignas(8) uint64_t bar_full[kGemmStages], bar_empty[kGemmStages], bar_acc_full[2], bar_acc_empty[2], bar_drain;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(GemmSmem) + 1024 <= 232448, "GEMM shared memory over the per-CTA limit");

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// TMA store of a {64 columns, 32 rows} box from shared memory (bulk group).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(src)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until the committed bulk stores have read their shared memory.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Waits until the committed bulk stores have completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Makes this thread's generic-proxy shared-memory writes visible to TMA.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y,
                                            int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// Loads one stage of an operand tile covering MN rows [mn0, mn0 + rows) and
// K [k0, k0 + 64). K-major: a 2-D box {64 K columns, rows}, landing as
// [row][128 B]. MN-major: a 3-D box {64 MN columns, 64 K rows, rows / 64
// groups}, landing as [group][K row][128 B]. x is 0 or k0, both multiples of
// 64 elements (128 bytes).
template <bool MN>
__device__ __forceinline__ void load_operand(uint32_t dst, const CUtensorMap* map, uint32_t bar, int mn0, int k0) {
  if (MN) tma_load_3d(dst, map, bar, 0, k0, mn0 / 64);
  else tma_load_2d(dst, map, bar, k0, mn0);
}

// Stores 32 bytes (eight words) at a 32-byte aligned address: a whole
// sector per store reaches L2 in one request.
__device__ __forceinline__ void store_words8(void* dst, const uint32_t* w) {
  asm volatile("st.global.L1::no_allocate.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(w[0]),
               "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

// Shared-memory descriptor of K-step kk (16 deep) of a stage tile.
template <bool MN>
__device__ __forceinline__ uint64_t operand_desc(uint32_t base, int kk) {
  if (MN) return sdesc_sw128(base + kk * 16 * 128, 64 * 128, 1024);  // LBO: between 64-wide MN groups
  return sdesc_sw128(base + kk * 32, 16, 1024);
}

template <typename T, bool A_MN, bool B_MN, int EPI>
__global__ void __launch_bounds__(kGemmThreads, 1) gemm_kernel(const __grid_constant__ GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  GemmSmem& s = *reinterpret_cast<GemmSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tm = (p.M + kGemmBM - 1) / kGemmBM, tn = (p.N + kGemmBN - 1) / kGemmBN;
  const int n_tiles = tm * tn * p.k_splits;
  const int nk_all = (p.K + kGemmBK - 1) / kGemmBK;
  const int per = (nk_all + p.k_splits - 1) / p.k_splits;
  // Tile t: K split t / (tm tn), then m tile, then n tile (fastest). Its K
  // blocks are [kb0, kb1) (empty only when k_splits exceeds the K blocks).
  auto tile_of = [&](int t, int& m0, int& n0, int& split, int& kb0, int& kb1) {
    split = t / (tm * tn);
    const int rem = t - split * tm * tn;
    m0 = (rem / tn) * kGemmBM;
    n0 = (rem % tn) * kGemmBN;
    kb0 = split * per;
    kb1 = kb0 + per < nk_all ? kb0 + per : nk_all;
    if (kb1 < kb0) kb1 = kb0;
  };
  constexpr uint32_t kStageBytes = (kGemmBM + kGemmBN) * kGemmBK * 2;
  if (threadIdx.x == 0) {
    s.abort_flag = 0;
    for (int i = 0; i < kGemmStages; ++i) {
      mbar_init(smem_u32(&s.bar_full[i]), 1);
      mbar_init(smem_u32(&s.bar_empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&s.bar_acc_full[i]), 1);
      mbar_init(smem_u32(&s.bar_acc_empty[i]), 128);  // the four epilogue warps
    }
    mbar_init(smem_u32(&s.bar_drain), 1);
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(&s.tmem_base), 2 * kGemmBN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = s.tmem_base;
  volatile int* abort_flag = &s.abort_flag;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&p.tm_a);
      tma_prefetch_map(&p.tm_b);
      int last[kGemmStages];
      for (int st = 0; st < kGemmStages; ++st) last[st] = -1;
      int g = 0;  // K blocks over all tiles of this CTA
      bool ok = true;
      for (int t = blockIdx.x; ok && t < n_tiles; t += gridDim.x) {
        int m0, n0, split, kb0, kb1;
        tile_of(t, m0, n0, split, kb0, kb1);
        for (int kb = kb0; kb < kb1; ++kb, ++g) {
          const int st = g % kGemmStages, use = g / kGemmStages;
          if (use > 0 && !mbar_wait(smem_u32(&s.bar_empty[st]), (use - 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t bar = smem_u32(&s.bar_full[st]);
          mbar_expect_tx(bar, kStageBytes);
          load_operand<A_MN>(smem_u32(s.a[st]), &p.tm_a, bar, m0, kb * kGemmBK);
          load_operand<B_MN>(smem_u32(s.b[st]), &p.tm_b, bar, n0, kb * kGemmBK);
          last[st] = use;
        }
      }
      for (int st = 0; st < kGemmStages; ++st)  // never leave with a copy in flight
        if (last[st] >= 0) mbar_wait_drain(smem_u32(&s.bar_full[st]), last[st] & 1);
    }
    __syncwarp();
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (elect_one_sync()) {
      constexpr uint32_t idesc = idesc_f16kind(kGemmBM, kGemmBN, A_MN, B_MN, Elem<T>::kUmma);
      int g = 0;  // K blocks over all tiles of this CTA
      int i = 0;  // tiles of this CTA
      bool ok = true;
      for (int t = blockIdx.x; ok && t < n_tiles; t += gridDim.x, ++i) {
        int m0, n0, split, kb0, kb1;
        tile_of(t, m0, n0, split, kb0, kb1);
        const int buf = i & 1;
        // accumulator buf is free once the epilogue has read out tile i - 2
        if (i >= 2 && !mbar_wait(smem_u32(&s.bar_acc_empty[buf]), ((i >> 1) - 1) & 1, abort_flag)) break;
        tc_fence_after();
        const uint32_t tacc = tbase + buf * kGemmBN;
        for (int kb = kb0; kb < kb1; ++kb, ++g) {
          const int st = g % kGemmStages;
          if (!mbar_wait(smem_u32(&s.bar_full[st]), (g / kGemmStages) & 1, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kGemmBK / 16; ++kk)
            umma_ss(tacc, operand_desc<A_MN>(smem_u32(s.a[st]), kk), operand_desc<B_MN>(smem_u32(s.b[st]), kk),
                    idesc, (kb > kb0 || kk > 0) ? 1u : 0u);
          umma_commit(smem_u32(&s.bar_empty[st]));
        }
        if (ok) umma_commit(smem_u32(&s.bar_acc_full[buf]));
      }
      umma_commit(smem_u32(&s.bar_drain));  // every MMA issued above has completed (also on abort)
      mbar_wait_drain(smem_u32(&s.bar_drain), 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    // Warp w reads TMEM lanes 32w.. (rows m0 + 32w + lane). fp32 partials
    // leave as 32-byte row stores; 16-bit outputs go through the warp's
    // staging buffers and leave as TMA stores of 32 rows x 64 columns, so
    // the global writes are whole 128-byte lines instead of a row a thread.
    const uint32_t lane_addr = static_cast<uint32_t>(warp * 32) << 16;
    const T* bias = static_cast<const T*>(p.bias);
    const uint32_t st_out = smem_u32(s.stage_out[warp]), st_out2 = smem_u32(s.stage_out2[warp]);
    const bool want2 = EPI == kEpiBiasSilu && p.out2 != nullptr;
    bool pending = false;  // lane 0: committed bulk stores may still read the staging buffers
    int i = 0;
    for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++i) {
      int m0, n0, split, kb0, kb1;
      tile_of(t, m0, n0, split, kb0, kb1);
      const int buf = i & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&s.bar_acc_full[buf]), (i >> 1) & 1, abort_flag))) break;
      tc_fence_after();
      const bool empty = kb1 == kb0;  // nothing accumulated: zeros
      const int row0 = m0 + warp * 32, row = row0 + lane;
      if (EPI == kEpiPartial) {
        for (int c = 0; c < kGemmBN / 32; ++c) {
          const int col = n0 + c * 32;
          uint32_t a[32];
          tmem_ld32(tbase + buf * kGemmBN + lane_addr + c * 32, a);
          tmem_ld_wait(a);
          if (empty)
#pragma unroll
            for (int e = 0; e < 32; ++e) a[e] = 0u;
          if (row >= p.M || col >= p.N) continue;  // N is a multiple of 32
          // fp32 rows of the workspace: always 32-byte aligned
          float* dst = p.partial + (static_cast<int64_t>(split) * p.M + row) * p.N + col;
#pragma unroll
          for (int e = 0; e < 4; ++e) store_words8(dst + 8 * e, a + 8 * e);
        }
      } else {
        for (int c = 0; c < kGemmBN / 64; ++c) {
          const int col = n0 + c * 64;
          // The chunk's 64 bias values (the same for every row): eight
          // 16-byte loads issued before the TMEM loads, so that both
          // latencies overlap.
          uint32_t bw[32];
          const bool live = col < p.N && row0 < p.M;  // warp-uniform; N is a multiple of 64
          if (EPI == kEpiBiasSilu && bias && live) {
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const uint4 v = *reinterpret_cast<const uint4*>(bias + col + 8 * q);
              bw[4 * q] = v.x;
              bw[4 * q + 1] = v.y;
              bw[4 * q + 2] = v.z;
              bw[4 * q + 3] = v.w;
            }
          } else {
#pragma unroll
            for (int q = 0; q < 32; ++q) bw[q] = 0u;
          }
          uint32_t a[32], b2[32];
          tmem_ld32(tbase + buf * kGemmBN + lane_addr + c * 64, a);
          tmem_ld32(tbase + buf * kGemmBN + lane_addr + c * 64 + 32, b2);
          tmem_ld_wait(a);
          tmem_ld_wait(b2);
          if (!live) continue;
          uint32_t pk[32], pz[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const uint32_t w0 = e < 16 ? a[2 * e] : b2[2 * e - 32];
            const uint32_t w1 = e < 16 ? a[2 * e + 1] : b2[2 * e - 31];
            float x0 = empty ? 0.0f : __uint_as_float(w0), x1 = empty ? 0.0f : __uint_as_float(w1);
            if (EPI == kEpiBiasSilu) {
              x0 += Elem<T>::lo(bw[e]);  // zero without a bias
              x1 += Elem<T>::hi(bw[e]);
              pz[e] = Elem<T>::pack2(x0, x1);
              // silu(x) = x/2 (1 + tanh(x/2)): one hardware tanh an element
              const float h0 = 0.5f * x0, h1 = 0.5f * x1;
              pk[e] = Elem<T>::pack2(fmaf(h0, tanh_approx(h0), h0), fmaf(h1, tanh_approx(h1), h1));
            } else {
              pk[e] = Elem<T>::pack2(x0, x1);
            }
          }
          // The previous chunk's stores must have read the staging buffers.
          if (lane == 0 && pending) bulk_wait_read_all();
          __syncwarp();
          // Row `lane`, 16-byte piece j lands at piece j ^ (lane & 7) of the
          // row (128-byte swizzle: conflict-free across each 8-row group).
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint32_t off = static_cast<uint32_t>(lane * 128 + ((j ^ (lane & 7)) << 4));
            st_shared_v4(st_out + off, pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
            if (want2) st_shared_v4(st_out2 + off, pz[4 * j], pz[4 * j + 1], pz[4 * j + 2], pz[4 * j + 3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {  // rows past M are clipped by the tensor map
            tma_store_2d(&p.tm_out, st_out, col, row0);
            if (want2) tma_store_2d(&p.tm_out2, st_out2, col, row0);
            bulk_commit();
            pending = true;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&s.bar_acc_empty[buf]));
    }
    if (lane == 0 && pending) bulk_wait_all();  // every store done before the CTA exits
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tbase, 2 * kGemmBN);
  }
  if (threadIdx.x == 0 && s.abort_flag && p.err) atomicOr(p.err, kErrTimeout);
}

// X_c[i] = x[rows[i]] (16-byte copies); a row index outside [0, x_rows)
// sets kErrInput and gives a zero row.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ x, int64_t x_rows,
                                                          const int32_t* __restrict__ rows, int64_t n,
                                                          int row_vecs, uint4* __restrict__ xc, int32_t* err) {
  const int64_t i = blockIdx.x;
  if (i >= n) return;
  const int r = rows[i];
  const bool ok = r >= 0 && r < x_rows;
  if (!ok && threadIdx.x == 0) atomicOr(err, kErrInput);
  for (int v = threadIdx.x; v < row_vecs; v += blockDim.x)
    xc[i * row_vecs + v] = ok ? x[static_cast<int64_t>(r) * row_vecs + v] : make_uint4(0, 0, 0, 0);
}

// G = dY * silu'(Z), eight consecutive columns a thread (16-byte loads and
// stores), and the bias gradient's partials: block b takes the row chunk
// [b R, (b + 1) R), R = ceil(rows / gridDim.x), and writes its column sums to
// part[b]. The threads of a block cover rpi = 256 / (cols / 8) rows of all
// columns per iteration when a row has at most 256 column groups, else one
// row of the 256 groups that gridDim.y picks; two rows are in flight per
// thread. Row lanes are summed in lane order through shared memory, so the
// partials are deterministic. cols is a multiple of 64.
template <typename T>
__global__ void __launch_bounds__(kGradThreads) silu_grad_kernel(const T* __restrict__ dy, const T* __restrict__ z,
                                                                 int64_t rows, int cols, T* __restrict__ g,
                                                                 float* __restrict__ part) {
  __shared__ float red[kGradThreads][8];
  const int groups = cols / 8;
  const int rpi = groups >= kGradThreads ? 1 : kGradThreads / groups;
  const int gy = groups >= kGradThreads ? kGradThreads : groups;  // column groups a block covers
  const int lane_row = threadIdx.x / gy, cg = blockIdx.y * gy + threadIdx.x % gy;
  const bool active = lane_row < rpi && cg < groups;
  const int col = cg * 8;
  const int64_t per = (rows + gridDim.x - 1) / gridDim.x;
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * per;
  const int64_t r1 = r0 + per < rows ? r0 + per : rows;
  float sum[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) sum[e] = 0.0f;
  auto grad_row = [&](const uint4& zv, const uint4& dv, int64_t idx) {
    const uint32_t zw[4] = {zv.x, zv.y, zv.z, zv.w}, dw[4] = {dv.x, dv.y, dv.z, dv.w};
    uint32_t gw[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float gv[2];
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        const float zz = x ? Elem<T>::hi(zw[e]) : Elem<T>::lo(zw[e]);
        const float d = x ? Elem<T>::hi(dw[e]) : Elem<T>::lo(dw[e]);
        const float sg = sigmoidf_fast(zz);
        gv[x] = d * sg * (1.0f + zz * (1.0f - sg));
      }
      gw[e] = Elem<T>::pack2(gv[0], gv[1]);
      // the bias gradient sums the same rounded G the GEMMs read
      sum[2 * e] += Elem<T>::lo(gw[e]);
      sum[2 * e + 1] += Elem<T>::hi(gw[e]);
    }
    *reinterpret_cast<uint4*>(g + idx) = make_uint4(gw[0], gw[1], gw[2], gw[3]);
  };
  if (active) {
    int64_t r = r0 + lane_row;
    for (; r + rpi < r1; r += 2 * rpi) {  // two rows in flight
      const int64_t i0 = r * cols + col, i1 = (r + rpi) * cols + col;
      const uint4 z0 = *reinterpret_cast<const uint4*>(z + i0), d0 = *reinterpret_cast<const uint4*>(dy + i0);
      const uint4 z1 = *reinterpret_cast<const uint4*>(z + i1), d1 = *reinterpret_cast<const uint4*>(dy + i1);
      grad_row(z0, d0, i0);
      grad_row(z1, d1, i1);
    }
    if (r < r1) {
      const int64_t i0 = r * cols + col;
      grad_row(*reinterpret_cast<const uint4*>(z + i0), *reinterpret_cast<const uint4*>(dy + i0), i0);
    }
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) red[threadIdx.x][e] = sum[e];
  __syncthreads();
  if (active && lane_row == 0) {
    float tot[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) tot[e] = 0.0f;
    for (int l = 0; l < rpi; ++l)
#pragma unroll
      for (int e = 0; e < 8; ++e) tot[e] += red[l * gy + threadIdx.x][e];
    float* dst = part + static_cast<int64_t>(blockIdx.x) * cols + col;
    reinterpret_cast<float4*>(dst)[0] = make_float4(tot[0], tot[1], tot[2], tot[3]);
    reinterpret_cast<float4*>(dst)[1] = make_float4(tot[4], tot[5], tot[6], tot[7]);
  }
}

// db[col] = sum of the chunk partials in chunk order: warp w of a block
// sums chunks w, w + 8, ... of 32 columns (a lane a column), then lane l of
// warp 0 adds the eight warps' sums in warp order.
template <typename T>
__global__ void __launch_bounds__(256) column_fold_kernel(const float* __restrict__ part, int chunks, int cols,
                                                          T* __restrict__ db) {
  __shared__ float red[8][32];
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  const int col = blockIdx.x * 32 + l;
  float s = 0.0f;
  if (col < cols)
    for (int c = w; c < chunks; c += 8) s += part[static_cast<int64_t>(c) * cols + col];
  red[w][l] = s;
  __syncthreads();
  if (w == 0 && col < cols) {
    float t = 0.0f;
#pragma unroll
    for (int x = 0; x < 8; ++x) t += red[x][l];
    const uint32_t word = Elem<T>::pack2(t, 0.0f);
    reinterpret_cast<uint16_t*>(db)[col] = static_cast<uint16_t>(word & 0xffffu);
  }
}

// out = sum over splits (in order) of the fp32 partials, 8 elements a thread.
template <typename T>
__global__ void __launch_bounds__(256) split_fold_kernel(const float* __restrict__ part, int splits, int64_t elems,
                                                         T* __restrict__ out) {
  const int64_t i = (static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x) * 8;
  if (i >= elems) return;
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
  for (int sp = 0; sp < splits; ++sp) {
    const float4* src = reinterpret_cast<const float4*>(part + sp * elems + i);
    const float4 a = src[0], b = src[1];
    acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
    acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
  }
  *reinterpret_cast<uint4*>(out + i) = make_uint4(Elem<T>::pack2(acc[0], acc[1]), Elem<T>::pack2(acc[2], acc[3]),
                                                 Elem<T>::pack2(acc[4], acc[5]), Elem<T>::pack2(acc[6], acc[7]));
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// Tensor map of a row-major (rows, cols) operand: K-major tiles are boxes of
// {64 columns, box_rows rows}; MN-major tiles are a 3-D view {64 columns,
// rows, cols / 64 groups} (group stride 128 B) with boxes {64, 64, box_cols /
// 64}. Rows or groups past the tensor read as zeros.
bool operand_map(CUtensorMap* m, const void* ptr, int64_t rows, int cols, int dtype, bool mn, int box_mn) {
  auto fn = encode_fn();
  if (!fn) return false;
  const CUtensorMapDataType type =
      dtype == HSTU_DTYPE_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const cuuint64_t row_bytes = static_cast<cuuint64_t>(cols) * 2;
  cuuint32_t es[3] = {1, 1, 1};
  if (!mn) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_mn)};
    return fn(m, type, 2, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  }
  cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(cols / 64)};
  cuuint64_t strides[2] = {row_bytes, 128};
  cuuint32_t box[3] = {64, 64, static_cast<cuuint32_t>(box_mn / 64)};
  return fn(m, type, 3, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename T, bool A_MN, bool B_MN, int EPI>
cudaError_t launch_gemm(const GemmParams& p_in, cudaStream_t stream) {
  GemmParams p = p_in;
  if (p.k_splits < 1) p.k_splits = 1;
  const int smem = static_cast<int>(sizeof(GemmSmem)) + 1024;
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (uint64_t{1} << dev) : 0;
  if (bit == 0 || (configured.load() & bit) == 0) {
    e = cudaFuncSetAttribute(gemm_kernel<T, A_MN, B_MN, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (bit) configured.fetch_or(bit);
  }
  const long long tiles = static_cast<long long>((p.M + kGemmBM - 1) / kGemmBM) * ((p.N + kGemmBN - 1) / kGemmBN) *
                          p.k_splits;
  if (tiles <= 0) return cudaSuccess;
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>(tiles < sms ? tiles : sms));  // persistent: one CTA per SM
  gemm_kernel<T, A_MN, B_MN, EPI><<<grid, kGemmThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Workspace of the projection: a 256-byte header (error word), then the
// gathered rows X_c (n x d_in), then (backward) G (n x d_out), the bias
// partials (grad_chunks(n) x d_out fp32) and the split-K partials of dW
// (kMaxKSplits x d_out x d_in fp32).
struct ProjLayout {
  size_t xc = 0, g = 0, part = 0, dwp = 0, total = 0;
};
ProjLayout proj_layout(int64_t n, int d_in, int d_out, bool bwd) {
  ProjLayout l;
  l.xc = kHdrWords * 4;
  l.g = l.xc + align_up(static_cast<size_t>(n) * d_in * 2, 256);
  l.part = l.g + (bwd ? align_up(static_cast<size_t>(n) * d_out * 2, 256) : 0);
  l.dwp = l.part + (bwd ? align_up(static_cast<size_t>(grad_chunks(n)) * d_out * 4, 256) : 0);
  l.total = l.dwp + (bwd ? align_up(static_cast<size_t>(kMaxKSplits) * d_out * d_in * 4, 256) : 0);
  return l;
}

hstu_status_t proj_checks(int64_t x_rows, int64_t n, int d_in, int d_out, int dtype) {
  if (x_rows < 0 || n < 0 || n > INT32_MAX || x_rows > INT32_MAX) return HSTU_ERR_INVALID_ARG;
  if (d_in < 64 || d_out < 64 || d_in % 64 || d_out % 64 || d_in > 65536 || d_out > 65536)
    return HSTU_ERR_UNSUPPORTED;
  if (dtype != HSTU_DTYPE_BF16 && dtype != HSTU_DTYPE_F16) return HSTU_ERR_UNSUPPORTED;
  return HSTU_OK;
}

template <typename T>
hstu_status_t project_fwd_t(const void* x, int64_t x_rows, const int32_t* rows, int64_t n, const void* w,
                            const void* bias, int d_in, int d_out, int dtype, void* y, void* z, void* ws,
                            cudaStream_t stream) {
  uint8_t* base = static_cast<uint8_t*>(ws);
  const ProjLayout l = proj_layout(rows ? n : 0, d_in, d_out, false);
  int32_t* err = reinterpret_cast<int32_t*>(base);
  if (cudaMemsetAsync(err, 0, kHdrWords * 4, stream) != cudaSuccess) return HSTU_ERR_CUDA;
  if (n == 0) return HSTU_OK;
  const void* a = x;
  if (rows) {
    gather_rows_kernel<<<static_cast<unsigned>(n), 256, 0, stream>>>(
        static_cast<const uint4*>(x), x_rows, rows, n, d_in / 8, reinterpret_cast<uint4*>(base + l.xc), err);
    if (cudaGetLastError() != cudaSuccess) return HSTU_ERR_CUDA;
    a = base + l.xc;
  }
  GemmParams p{};
  if (!operand_map(&p.tm_a, a, n, d_in, dtype, false, kGemmBM) ||
      !operand_map(&p.tm_b, w, d_out, d_in, dtype, false, kGemmBN))
    return HSTU_ERR_CUDA;
  p.out = y;
  p.out2 = z;
  if (!operand_map(&p.tm_out, y, n, d_out, dtype, false, 32) ||
      (z && !operand_map(&p.tm_out2, z, n, d_out, dtype, false, 32)))
    return HSTU_ERR_CUDA;
  p.bias = bias;
  p.err = err;
  p.M = static_cast<int32_t>(n);
  p.N = d_out;
  p.K = d_in;
  p.ldo = d_out;
  return launch_gemm<T, false, false, kEpiBiasSilu>(p, stream) == cudaSuccess ? HSTU_OK : HSTU_ERR_CUDA;
}

template <typename T>
hstu_status_t project_bwd_t(const void* dy, const void* z, const void* x, int64_t x_rows, const int32_t* rows,
                            int64_t n, const void* w, int d_in, int d_out, int dtype, void* dx_c, void* dw,
                            void* dbias, void* ws, cudaStream_t stream) {
  uint8_t* base = static_cast<uint8_t*>(ws);
  const ProjLayout l = proj_layout(n, d_in, d_out, true);
  int32_t* err = reinterpret_cast<int32_t*>(base);
  if (cudaMemsetAsync(err, 0, kHdrWords * 4, stream) != cudaSuccess) return HSTU_ERR_CUDA;
  if (n == 0) {  // no rows: dW and db are zero
    if (cudaMemsetAsync(dw, 0, static_cast<size_t>(d_out) * d_in * 2, stream) != cudaSuccess) return HSTU_ERR_CUDA;
    if (dbias && cudaMemsetAsync(dbias, 0, static_cast<size_t>(d_out) * 2, stream) != cudaSuccess)
      return HSTU_ERR_CUDA;
    return HSTU_OK;
  }
  T* g = reinterpret_cast<T*>(base + l.g);
  float* part = reinterpret_cast<float*>(base + l.part);
  const int chunks = grad_chunks(n);
  silu_grad_kernel<T><<<dim3(chunks, (d_out / 8 + kGradThreads - 1) / kGradThreads), kGradThreads, 0, stream>>>(
      static_cast<const T*>(dy), static_cast<const T*>(z), n, d_out, g, part);
  if (cudaGetLastError() != cudaSuccess) return HSTU_ERR_CUDA;
  if (dbias) {
    column_fold_kernel<T><<<(d_out + 31) / 32, 256, 0, stream>>>(part, chunks, d_out, static_cast<T*>(dbias));
    if (cudaGetLastError() != cudaSuccess) return HSTU_ERR_CUDA;
  }
  const void* xc = x;
  if (rows) {
    gather_rows_kernel<<<static_cast<unsigned>(n), 256, 0, stream>>>(
        static_cast<const uint4*>(x), x_rows, rows, n, d_in / 8, reinterpret_cast<uint4*>(base + l.xc), err);
    if (cudaGetLastError() != cudaSuccess) return HSTU_ERR_CUDA;
    xc = base + l.xc;
  }
  // dX_c (n x d_in) = G (n x d_out, K-major) . W (d_out x d_in read MN-major: N = d_in, K = d_out)
  GemmParams p1{};
  if (!operand_map(&p1.tm_a, g, n, d_out, dtype, false, kGemmBM) ||
      !operand_map(&p1.tm_b, w, d_out, d_in, dtype, true, kGemmBN))
    return HSTU_ERR_CUDA;
  p1.out = dx_c;
  if (!operand_map(&p1.tm_out, dx_c, n, d_in, dtype, false, 32)) return HSTU_ERR_CUDA;
  p1.err = err;
  p1.M = static_cast<int32_t>(n);
  p1.N = d_in;
  p1.K = d_out;
  p1.ldo = d_in;
  if (launch_gemm<T, false, true, kEpiStore>(p1, stream) != cudaSuccess) return HSTU_ERR_CUDA;
  // dW (d_out x d_in) = G^T (M = d_out, K = n: MN-major) . X_c (N = d_in, K = n: MN-major)
  GemmParams p2{};
  if (!operand_map(&p2.tm_a, g, n, d_out, dtype, true, kGemmBM) ||
      !operand_map(&p2.tm_b, xc, n, d_in, dtype, true, kGemmBN))
    return HSTU_ERR_CUDA;
  p2.out = dw;
  if (!operand_map(&p2.tm_out, dw, d_out, d_in, dtype, false, 32)) return HSTU_ERR_CUDA;
  p2.err = err;
  p2.M = d_out;
  p2.N = d_in;
  p2.K = static_cast<int32_t>(n);
  p2.ldo = d_in;
  // K (the rows) is long and the output has few tiles: split K so that the
  // grid covers the SMs twice, then fold the fp32 partials in split order.
  const int tiles = ((d_out + kGemmBM - 1) / kGemmBM) * ((d_in + kGemmBN - 1) / kGemmBN);
  const int nk = static_cast<int>((n + kGemmBK - 1) / kGemmBK);
  int splits = (2 * 152 + tiles - 1) / tiles;
  splits = splits < 1 ? 1 : (splits > kMaxKSplits ? kMaxKSplits : splits);
  splits = splits > nk ? nk : splits;
  if (splits <= 1) return launch_gemm<T, true, true, kEpiStore>(p2, stream) == cudaSuccess ? HSTU_OK : HSTU_ERR_CUDA;
  p2.k_splits = splits;
  p2.partial = reinterpret_cast<float*>(base + l.dwp);
  if (launch_gemm<T, true, true, kEpiPartial>(p2, stream) != cudaSuccess) return HSTU_ERR_CUDA;
  const int64_t elems = static_cast<int64_t>(d_out) * d_in;
  split_fold_kernel<T><<<static_cast<unsigned>((elems / 8 + 255) / 256), 256, 0, stream>>>(p2.partial, splits, elems,
                                                                                          static_cast<T*>(dw));
  return cudaGetLastError() == cudaSuccess ? HSTU_OK : HSTU_ERR_CUDA;
}

}  // namespace
}  // namespace hstu

extern "C" {

HSTU_API size_t hstu_attn_project_workspace_size(int64_t num_rows, int32_t d_in, int32_t d_out, int32_t backward) {
  if (hstu::proj_checks(0, num_rows, d_in, d_out, HSTU_DTYPE_BF16) != HSTU_OK) return 0;
  return hstu::proj_layout(num_rows, d_in, d_out, backward != 0).total;
}

HSTU_API hstu_status_t hstu_attn_project_rows(const void* x, int64_t x_rows, const int32_t* rows, int64_t num_rows,
                                              const void* w, const void* bias, int32_t d_in, int32_t d_out,
                                              int32_t dtype, void* y, void* z, void* ws, size_t ws_bytes,
                                              void* stream) {
  hstu_status_t st = hstu::proj_checks(x_rows, num_rows, d_in, d_out, dtype);
  if (st != HSTU_OK) return st;
  if (!rows && num_rows != x_rows) return HSTU_ERR_INVALID_ARG;
  if (num_rows > 0 && (!hstu::aligned16(x) || !hstu::aligned16(w) || !hstu::aligned16(y) ||
                       (z && !hstu::aligned16(z)) || (bias && !hstu::aligned16(bias))))
    return HSTU_ERR_INVALID_ARG;
  if (rows && (reinterpret_cast<uintptr_t>(rows) & 3u)) return HSTU_ERR_INVALID_ARG;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) ||
      ws_bytes < hstu_attn_project_workspace_size(rows ? num_rows : 0, d_in, d_out, 0))
    return HSTU_ERR_WORKSPACE;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  return dtype == HSTU_DTYPE_F16
             ? hstu::project_fwd_t<__half>(x, x_rows, rows, num_rows, w, bias, d_in, d_out, dtype, y, z, ws, cs)
             : hstu::project_fwd_t<__nv_bfloat16>(x, x_rows, rows, num_rows, w, bias, d_in, d_out, dtype, y, z,
                                                  ws, cs);
}

HSTU_API hstu_status_t hstu_attn_project_rows_bwd(const void* dy, const void* z, const void* x, int64_t x_rows,
                                                  const int32_t* rows, int64_t num_rows, const void* w,
                                                  int32_t d_in, int32_t d_out, int32_t dtype, void* dx_rows,
                                                  void* dw, void* dbias, void* ws, size_t ws_bytes, void* stream) {
  hstu_status_t st = hstu::proj_checks(x_rows, num_rows, d_in, d_out, dtype);
  if (st != HSTU_OK) return st;
  if (!rows && num_rows != x_rows) return HSTU_ERR_INVALID_ARG;
  if (!hstu::aligned16(dw) || !dw) return HSTU_ERR_INVALID_ARG;
  if (num_rows > 0 && (!hstu::aligned16(dy) || !hstu::aligned16(z) || !hstu::aligned16(x) ||
                       !hstu::aligned16(w) || !hstu::aligned16(dx_rows) || !dy || !z || !x || !w || !dx_rows))
    return HSTU_ERR_INVALID_ARG;
  if ((rows && (reinterpret_cast<uintptr_t>(rows) & 3u)) || (dbias && (reinterpret_cast<uintptr_t>(dbias) & 3u)))
    return HSTU_ERR_INVALID_ARG;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) ||
      ws_bytes < hstu_attn_project_workspace_size(num_rows, d_in, d_out, 1))
    return HSTU_ERR_WORKSPACE;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  return dtype == HSTU_DTYPE_F16
             ? hstu::project_bwd_t<__half>(dy, z, x, x_rows, rows, num_rows, w, d_in, d_out, dtype, dx_rows, dw,
                                           dbias, ws, cs)
             : hstu::project_bwd_t<__nv_bfloat16>(dy, z, x, x_rows, rows, num_rows, w, d_in, d_out, dtype, dx_rows,
                                                  dw, dbias, ws, cs);
}

}  // extern "C"
