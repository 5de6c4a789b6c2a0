// Plan: device-side validation of seq_offsets, the func prologue that
// classifies every (q-tile, kv-tile) pair of a sequence, the per-row visible
// counts, and the longest-first work lists of the forward and backward
// kernels, all in one launch. Nothing here needs a host synchronisation.
// The work lists depend on seq_offsets alone, so block 0 validates the
// offsets and builds them while the other blocks classify tiles; block 0 also
// writes every header word the kernels read, so no memset precedes the plan.
//
// The pages' kernels reduce per-tile min/max bounds of every interval
// (including the empty padded ones) and then test every interval in every KV
// block (TorchEasyRec PR #670, review thread: the cost of the padded third
// interval came from those reductions and from the per-block masking loop).
// Here empty intervals are normalised away before anything else, and each
// pair's class comes from exact per-row popcounts of the row's visible
// columns inside the tile:
//   skip    -- no valid row sees any column of the tile,
//   full    -- every row of the q tile is valid and sees all 128 columns,
//   partial -- anything else (the kernels then apply the per-row mask).
// A partial pair also records which 64-wide halves are dead: the kv half no
// row sees (kLoKvDead / kHiKvDead) and the q half that sees no column of the
// tile (kLoQDead / kHiQDead). The kernels skip the MMAs and the epilogue of a
// dead half; on a causal window of 32 columns that saves one half-tile of
// every four.
#include "common.cuh"
#include "internal.h"

namespace hstu {

// Classifies the kv tiles seen by one (sequence b, q tile qt) block and
// writes that tile's row counts, class row and active-interval mask. Blocks
// past a sequence's last q tile (or of an invalid sequence, which block 0
// reports) do nothing.
template <int NINT>
__device__ void classify_tile(const PlanParams& p, int b, int qt) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int o0 = p.seq_offsets[b];
  const int o1 = p.seq_offsets[b + 1];
  const int L = o1 - o0;
  if (L < 0 || L > p.max_seqlen || o0 < 0 || static_cast<int64_t>(o1) > p.total) return;
  const int ntiles = (L + kBlock - 1) / kBlock;
  if (qt >= ntiles) return;

  // Per warp (32 rows) and kv tile: some row sees kv columns 0..63 (lo),
  // 64..127 (hi); every row sees all 128 (all).
  __shared__ uint32_t all_bits[4][kMaxTiles / 32];
  __shared__ uint32_t lo_bits[4][kMaxTiles / 32];
  __shared__ uint32_t hi_bits[4][kMaxTiles / 32];
  __shared__ uint32_t active_iv;
  if (tid == 0) active_iv = 0;
  for (int x = tid; x < 4 * (kMaxTiles / 32); x += 128) {
    (&all_bits[0][0])[x] = 0;
    (&lo_bits[0][0])[x] = 0;
    (&hi_bits[0][0])[x] = 0;
  }
  __syncthreads();

  const int i = qt * kBlock + tid;
  const bool valid = i < L;
  int lo[NINT], hi[NINT];
  load_row_intervals<NINT>(p.func, p.total, static_cast<int64_t>(o0) + i, L, valid, lo, hi);
  uint32_t nonempty = 0;
#pragma unroll
  for (int t = 0; t < NINT; ++t) nonempty |= (hi[t] > lo[t] ? 1u : 0u) << t;
  nonempty = __reduce_or_sync(0xffffffffu, nonempty);
  if (lane == 0 && nonempty) atomicOr(&active_iv, nonempty);

  // No row of this warp sees a column at or past its largest interval end:
  // the kv tiles from there on are skip for the warp (their bits stay 0).
  int hi_row = 0;
#pragma unroll
  for (int t = 0; t < NINT; ++t) hi_row = max(hi_row, hi[t]);
  const int hi_warp = __reduce_max_sync(0xffffffffu, hi_row);
  const int jmax = min(ntiles, (hi_warp + kBlock - 1) / kBlock);
  int count = 0;
  for (int j = 0; j < jmax; ++j) {
    // Most tiles lie wholly inside one interval or outside all of them (an
    // empty interval is [0,0) and never meets a tile); only the others need
    // the row's column bits.
    const int s0 = j * kBlock;
    bool none = true, cover = false;
#pragma unroll
    for (int t = 0; t < NINT; ++t) {
      none = none && (hi[t] <= s0 || lo[t] >= s0 + kBlock);
      cover = cover || (lo[t] <= s0 && hi[t] >= s0 + kBlock);
    }
    int c_lo = cover ? kBlock / 2 : 0, c_hi = c_lo;
    if (!cover && !none) {
      c_lo = __popc(row_mask_word<NINT>(lo, hi, s0)) + __popc(row_mask_word<NINT>(lo, hi, s0 + 32));
      c_hi = __popc(row_mask_word<NINT>(lo, hi, s0 + 64)) + __popc(row_mask_word<NINT>(lo, hi, s0 + 96));
    }
    const int c = c_lo + c_hi;
    count += c;
    const unsigned all = __ballot_sync(0xffffffffu, c == kBlock);
    const unsigned any_lo = __ballot_sync(0xffffffffu, c_lo > 0);
    const unsigned any_hi = __ballot_sync(0xffffffffu, c_hi > 0);
    if (lane == 0) {
      const uint32_t bit = 1u << (j & 31);
      if (all == 0xffffffffu) all_bits[warp][j >> 5] |= bit;
      if (any_lo) lo_bits[warp][j >> 5] |= bit;
      if (any_hi) hi_bits[warp][j >> 5] |= bit;
    }
  }
  if (valid && p.row_counts) p.row_counts[o0 + i] = count;
  __syncthreads();

  const size_t row_base = (static_cast<size_t>(b) * p.nt + qt) * p.nt;
  for (int j = tid; j < ntiles; j += 128) {
    const uint32_t bit = 1u << (j & 31);
    const int word = j >> 5;
    uint32_t wany[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) wany[w] = lo_bits[w][word] | hi_bits[w][word];
    const bool any = ((wany[0] | wany[1] | wany[2] | wany[3]) & bit) != 0;
    const bool all = ((all_bits[0][word] & all_bits[1][word] & all_bits[2][word] &
                       all_bits[3][word]) & bit) != 0;
    uint8_t c = all ? kFull : (any ? kPartial : kSkip);
    if (c == kPartial) {
      const uint32_t lo_kv = lo_bits[0][word] | lo_bits[1][word] | lo_bits[2][word] | lo_bits[3][word];
      const uint32_t hi_kv = hi_bits[0][word] | hi_bits[1][word] | hi_bits[2][word] | hi_bits[3][word];
      if (!(lo_kv & bit)) c |= kLoKvDead;
      if (!(hi_kv & bit)) c |= kHiKvDead;
      if (!((wany[0] | wany[1]) & bit)) c |= kLoQDead;  // q rows 0..63
      if (!((wany[2] | wany[3]) & bit)) c |= kHiQDead;  // q rows 64..127
    }
    p.cls[row_base + j] = c;
  }
  if (tid == 0) p.ivmask[static_cast<size_t>(b) * p.nt + qt] = static_cast<uint8_t>(active_iv);
}

// Work lists. Sequences are ordered longest first (a counting sort on their
// tile count) and every sequence's items are contiguous, so the CTAs that
// run at the same time work on one or two sequences and share their K/V (or
// Q/dO) tiles in L2 instead of streaming every sequence's tiles from HBM at
// once. Within a sequence the heaviest items come first: forward q tiles
// last-first (the later rows of causal-like masks see the most columns);
// backward dK/dV kv tiles first-first and dQ q tiles last-first, the two
// roles grouped in windows of list entries (below). Sequences of equal tile
// count may come out in any order: every output element is computed by
// exactly one CTA with a fixed internal order, so the order only changes
// scheduling, never results.
//
// Block 0 does this in two passes over the sequences, each thread keeping
// kListUnroll sequences' offset loads in flight:
//   1. check seq_offsets (first 0, last = total, every length in
//      [0, max_seqlen]) and count the sequences of each tile count (bin
//      nt - tiles, so that bins run longest first), one shared atomic per
//      bin and warp;
//   2. give each sequence its position within its bin (again one atomic per
//      bin and warp) and write its items. The sequences before it are the
//      earlier bins and the earlier positions of its own bin, so its first
//      list entry follows from the bins' prefix sums without a scan over
//      the batch.
// It writes the header: the error word (kErrInput, with empty lists, if the
// check fails), the list lengths, the uniform flag and the zeroed work
// counters.
constexpr int kListUnroll = 8;

__device__ void build_work_lists(const PlanParams& p) {
  __shared__ int hist[kMaxTiles + 1];      // sequences per bin
  __shared__ int bin_pos[kMaxTiles + 1];   // first sorted position of each bin
  __shared__ int bin_item[kMaxTiles + 1];  // first list entry of each bin
  __shared__ int cursor[kMaxTiles + 1];    // next free position of each bin
  __shared__ int n_items, n_first, uniform_s, bad;
  const int tid = threadIdx.x, lane = tid & 31;
  const int nt = p.nt;
  const int step = kListUnroll * static_cast<int>(blockDim.x);
  // The sequences of this thread in one round of a pass, their offsets, and
  // their bins (-1 past the batch).
  auto load_round = [&](int base, int (&o0)[kListUnroll], int (&o1)[kListUnroll]) {
#pragma unroll
    for (int u = 0; u < kListUnroll; ++u) {
      const int b = base + u * static_cast<int>(blockDim.x) + tid;
      o0[u] = b < p.batch ? p.seq_offsets[b] : 0;
      o1[u] = b < p.batch ? p.seq_offsets[b + 1] : 0;
    }
  };
  auto bin_of = [&](int o0, int o1) {
    int64_t L = static_cast<int64_t>(o1) - o0;
    L = L < 0 ? 0 : (L > p.max_seqlen ? p.max_seqlen : L);
    return nt - static_cast<int>((L + kBlock - 1) / kBlock);
  };

  if (tid == 0)
    bad = (p.seq_offsets[0] != 0 || static_cast<int64_t>(p.seq_offsets[p.batch]) != p.total) ? 1 : 0;
  for (int x = tid; x <= nt; x += blockDim.x) hist[x] = 0;
  __syncthreads();
  for (int base = 0; base < p.batch; base += step) {
    int o0[kListUnroll], o1[kListUnroll];
    load_round(base, o0, o1);
#pragma unroll
    for (int u = 0; u < kListUnroll; ++u) {
      const int b = base + u * static_cast<int>(blockDim.x) + tid;
      int bin = -1;
      if (b < p.batch) {
        const int64_t L = static_cast<int64_t>(o1[u]) - o0[u];
        if (o0[u] < 0 || static_cast<int64_t>(o1[u]) > p.total || L < 0 || L > p.max_seqlen)
          bad = 1;  // every writer stores the same value
        bin = bin_of(o0[u], o1[u]);
      }
      const unsigned same = __match_any_sync(0xffffffffu, bin);
      if (bin >= 0 && lane == __ffs(same) - 1) atomicAdd(&hist[bin], __popc(same));
    }
  }
  __syncthreads();
  if (tid == 0) {
    p.header[kHdrFwdNext] = 0;
    p.header[kHdrFwdDone] = 0;
    p.header[kHdrBwdNext] = 0;
    p.header[kHdrBwdDone] = 0;
  }
  if (bad) {
    if (tid == 0) {
      p.header[kHdrErr] = kErrInput;
      p.header[kHdrNFwd] = 0;
      p.header[kHdrNBwd] = 0;
      p.header[kHdrUniform] = 0;
    }
    return;
  }
  if (tid == 0) {
    int pos = 0, item = 0, first = -1, last = -1;
    for (int x = 0; x <= nt; ++x) {
      bin_pos[x] = pos;
      cursor[x] = pos;
      bin_item[x] = item;
      if (hist[x] > 0) {
        if (first < 0) first = x;
        last = x;
      }
      pos += hist[x];
      item += hist[x] * (nt - x);
    }
    n_items = item;
    n_first = nt - first;           // the longest sequence's tile count (batch >= 1)
    uniform_s = first == last ? 1 : 0;  // every sequence has that many tiles
  }
  __syncthreads();
  // Backward: entry e = st + t of the sequence-major order goes to window
  // w = e / role_window; a window lists its dK/dV items first, then its dQ
  // items (the dQ item paired with kv tile t is q tile n - 1 - t). A CTA
  // then runs a few items of one role before the other, and a dQ item
  // seldom follows a dK/dV item, whose accumulator read-out it would wait
  // for; the window is sized so that its sequences' tiles stay in L2.
  // Batches whose sequences all have the same tile count n use windows of
  // n, one sequence each (its dK/dV items, then its dQ items): their CTAs
  // take items by a fixed stride, which balances that order by
  // construction, and a window spanning sequences can unbalance it.
  const int total = n_items, win = uniform_s ? max(n_first, 1) : p.role_window;
  for (int base = 0; base < p.batch; base += step) {
    int o0[kListUnroll], o1[kListUnroll];
    load_round(base, o0, o1);
#pragma unroll
    for (int u = 0; u < kListUnroll; ++u) {
      const int b = base + u * static_cast<int>(blockDim.x) + tid;
      const int bin = b < p.batch ? bin_of(o0[u], o1[u]) : -1;
      const unsigned same = __match_any_sync(0xffffffffu, bin);
      const int leader = __ffs(same) - 1;
      int first_pos = 0;
      if (bin >= 0 && lane == leader) first_pos = atomicAdd(&cursor[bin], __popc(same));
      first_pos = __shfl_sync(0xffffffffu, first_pos, leader);
      if (bin < 0) continue;
      const int pos = first_pos + __popc(same & ((1u << lane) - 1u));
      const int n = nt - bin;
      const int st = bin_item[bin] + (pos - bin_pos[bin]) * n;
      // Entry e = st + t lies at r = e - w0 in the window starting at w0,
      // which holds len entries of each role; both advance with e.
      int w0 = st / win * win, r = st - w0, len = min(win, total - w0);
      for (int t = 0; t < n; ++t) {
        p.fwd_list[st + t] = (b << 8) | (n - 1 - t);
        p.bwd_list[2 * w0 + r] = (b << 8) | t | kRoleDkdv;
        p.bwd_list[2 * w0 + len + r] = (b << 8) | (n - 1 - t);
        if (++r == win) {
          w0 += win;
          r = 0;
          len = min(win, total - w0);
        }
      }
    }
  }
  if (tid == 0) {
    p.header[kHdrErr] = 0;
    p.header[kHdrNFwd] = n_items;
    p.header[kHdrNBwd] = 2 * n_items;
    p.header[kHdrUniform] = uniform_s;
  }
}

// One launch of 1 + batch * nt blocks: block 0 checks the offsets and builds
// the work lists; block 1 + b * nt + qt classifies (sequence b, q tile qt).
template <int NINT>
__global__ void __launch_bounds__(128) plan_kernel(const PlanParams p) {
  if (blockIdx.x == 0) {
    build_work_lists(p);
    return;
  }
  const int idx = static_cast<int>(blockIdx.x) - 1;
  classify_tile<NINT>(p, idx / p.nt, idx % p.nt);
}

cudaError_t launch_plan(const PlanParams& p, cudaStream_t stream) {
  const long long blocks = 1 + static_cast<long long>(p.batch) * p.nt;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const unsigned grid = static_cast<unsigned>(blocks);
  const int nint = (p.nfunc + 1) / 2;
  switch (nint) {
    case 1: plan_kernel<1><<<grid, 128, 0, stream>>>(p); break;
    case 2: plan_kernel<2><<<grid, 128, 0, stream>>>(p); break;
    case 3: plan_kernel<3><<<grid, 128, 0, stream>>>(p); break;
    case 4: plan_kernel<4><<<grid, 128, 0, stream>>>(p); break;
    default: plan_kernel<5><<<grid, 128, 0, stream>>>(p); break;
  }
  return cudaGetLastError();
}

}  // namespace hstu
