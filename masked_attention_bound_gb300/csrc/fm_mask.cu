// Mask analysis on the device: per-k-block bound summary, tile classification
// with compacted work lists, the longest-first unit order, and localisation of
// the bounds to a rank's query chunks.  All integer work; bit-exact by design.
#include <climits>

#include "fm_internal.h"
#include "fm_ptx.cuh"

namespace fm {

// ------------------------------------------------------------------ summary
// One CTA per (k-block, batch*mask-head); one thread per key column.
// summary[(bh*nK + kj)*8 + ...] = min/max of LTS, LTE, UTS, UTE over the
// block's valid columns.  Any bound outside [0, Sq] sets DEV_BOUNDS.
__global__ void __launch_bounds__(kTile) summary_kernel(const int32_t* __restrict__ lts,
                                                        const int32_t* __restrict__ lte,
                                                        const int32_t* __restrict__ uts,
                                                        const int32_t* __restrict__ ute, int Sq,
                                                        int Skv, int nK, int32_t* summary,
                                                        int* status) {
  const int kj = blockIdx.x, bh = blockIdx.y;
  const int j = kj * kTile + threadIdx.x;
  int mn[4], mx[4];
  if (j < Skv) {
    const size_t at = static_cast<size_t>(bh) * Skv + j;
    const int v[4] = {__ldg(lts + at), __ldg(lte + at), __ldg(uts + at), __ldg(ute + at)};
    bool bad = false;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      mn[t] = mx[t] = v[t];
      bad |= (v[t] < 0) | (v[t] > Sq);
    }
    if (bad) atomicOr(status, DEV_BOUNDS);
  } else {
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      mn[t] = INT_MAX;
      mx[t] = INT_MIN;
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      mn[t] = min(mn[t], __shfl_xor_sync(0xffffffffu, mn[t], off));
      mx[t] = max(mx[t], __shfl_xor_sync(0xffffffffu, mx[t], off));
    }
  }
  __shared__ int red[kTile / 32][8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      red[warp][2 * t] = mn[t];
      red[warp][2 * t + 1] = mx[t];
    }
  }
  __syncthreads();
  if (threadIdx.x < 8) {
    const int t = threadIdx.x;
    int r = red[0][t];
    for (int w = 1; w < kTile / 32; ++w) r = (t & 1) ? max(r, red[w][t]) : min(r, red[w][t]);
    summary[(static_cast<size_t>(bh) * nK + kj) * 8 + t] = r;
  }
}

// ------------------------------------------------------------------ classify
// The tile rule for rows [r0, r1), r1 = min(r0 + 128, Sq), from one k-block's
// summary s = {minLTS, maxLTS, minLTE, maxLTE, minUTS, maxUTS, minUTE, maxUTE}.
__device__ __forceinline__ int classify(const int* s, int r0, int r1) {
  const bool cover_l = (s[1] <= r0) & (s[2] >= r1);
  const bool cover_u = (s[5] <= r0) & (s[6] >= r1);
  const bool miss_l = (s[0] >= r1) | (s[3] <= r0);
  const bool miss_u = (s[4] >= r1) | (s[7] <= r0);
  return (cover_l | cover_u) ? CLS_EMPTY : ((miss_l & miss_u) ? CLS_FULL : CLS_PARTIAL);
}

__device__ __forceinline__ void load_summary(const int32_t* p, int* s) {
  const int4 a = *reinterpret_cast<const int4*>(p);
  const int4 b = *reinterpret_cast<const int4*>(p + 4);
  s[0] = a.x; s[1] = a.y; s[2] = a.z; s[3] = a.w;
  s[4] = b.x; s[5] = b.y; s[6] = b.z; s[7] = b.w;
}

// One warp per (bh, q-tile): writes the table row and the ascending list of
// non-empty k-tiles, compacted with a ballot so the order is preserved.
// It also counts the row's tiles that take the element-wise path (class
// PARTIAL, or the ragged last key tile) and reserves that many consecutive
// slots of the visibility-mask region (row_mask = first slot, -1 if none or
// if the region is full: the forward then builds those tiles' bits itself).
__device__ __forceinline__ void classify_row(int w, const int32_t* __restrict__ summary, int nBH,
                                             int nQ, int nK, int Sq, int Skv, uint8_t* table,
                                             int32_t* row_count, int32_t* row_list,
                                             int32_t* row_mask, unsigned long long* slot_counter,
                                             int mask_cap) {
  const int lane = threadIdx.x & 31;
  if (w >= nBH * nQ) return;
  const int bh = w / nQ, qi = w - bh * nQ;
  const int r0 = qi * kTile, r1 = min(r0 + kTile, Sq);
  const int32_t* sm = summary + static_cast<size_t>(bh) * nK * 8;
  uint8_t* tab = table + static_cast<size_t>(w) * nK;
  int32_t* lst = row_list + static_cast<size_t>(w) * nK;
  const unsigned lt_mask = (1u << lane) - 1u;
  const bool ragged = (Skv & (kTile - 1)) != 0;
  int cnt = 0, npart = 0;
  for (int base = 0; base < nK; base += 32) {
    const int kj = base + lane;
    int cls = CLS_EMPTY;
    if (kj < nK) {
      int s[8];
      load_summary(sm + kj * 8, s);
      cls = classify(s, r0, r1);
      tab[kj] = static_cast<uint8_t>(cls);
    }
    const unsigned m = __ballot_sync(0xffffffffu, cls != CLS_EMPTY);
    if (cls != CLS_EMPTY) lst[cnt + __popc(m & lt_mask)] = (kj << 2) | cls;
    cnt += __popc(m);
    npart += __popc(__ballot_sync(0xffffffffu, cls == CLS_PARTIAL ||
                                                   (cls != CLS_EMPTY && ragged && kj == nK - 1)));
  }
  if (lane == 0) {
    row_count[w] = cnt;
    int first = -1;
    if (npart > 0 && mask_cap > 0) {
      const unsigned long long at = atomicAdd(slot_counter, static_cast<unsigned long long>(npart));
      if (at + static_cast<unsigned long long>(npart) <= static_cast<unsigned long long>(mask_cap))
        first = static_cast<int>(at);
    }
    row_mask[w] = first;
  }
}

// Visibility bit masks of the partial tiles of one q-tile row (one CTA per
// row, thread r = query row r0 + r of the tile): bit c of row r is set when
// key column kj*128 + c is hidden from that row (or lies past Skv).  The
// masks depend only on (batch, mask head), so every query head reuses them.
// kMaskSplit CTAs share a row (blockIdx.y = g builds the row's partial
// tiles g, g + kMaskSplit, ...), so a row with many partial tiles does not
// set the kernel's length.  Each reads the row's tile list in coalesced
// chunks and compacts the partial tiles in shared memory; the bounds of its
// tiles are loaded kMaskBatch tiles at a time (one load latency per batch),
// each thread reading column r of every tile of the batch.
constexpr int kMaskBatch = 4, kMaskSplit = 8;
__global__ void __launch_bounds__(kTile) tile_mask_kernel(
    const int32_t* __restrict__ lts, const int32_t* __restrict__ lte,
    const int32_t* __restrict__ uts, const int32_t* __restrict__ ute, int nQ, int nK, int Skv,
    const int32_t* __restrict__ row_count, const int32_t* __restrict__ row_list,
    const int32_t* __restrict__ row_mask, uint4* masks) {
  __shared__ int4 sb[kMaskBatch][kTile];
  __shared__ int kjs[kTile];   // partial tiles of the current list chunk, in list order
  __shared__ int nchunk_part;
  __shared__ int warp_part[kTile / 32];
  const int row = blockIdx.x;
  const int first = row_mask[row];
  if (first < 0) return;
  const int bh = row / nQ, qi = row - bh * nQ;
  const int n = row_count[row];
  const int32_t* lst = row_list + static_cast<size_t>(row) * nK;
  const size_t bbase = static_cast<size_t>(bh) * Skv;
  const int r = threadIdx.x, lane = r & 31, wid = r >> 5;
  const int R = qi * kTile + r;
  const bool ragged = (Skv & (kTile - 1)) != 0;
  int ord = 0;  // partial tiles written so far
  for (int base = 0; base < n; base += kTile) {
    // compact this chunk's partial tiles, keeping list order
    const int t = base + r;
    bool part = false;
    int kj = 0;
    if (t < n) {
      const int e = lst[t];
      kj = e >> 2;
      part = (e & 3) == CLS_PARTIAL || (ragged && kj == nK - 1);
    }
    const unsigned m = __ballot_sync(0xffffffffu, part);
    __syncthreads();  // the previous chunk's kjs and bounds are no longer read
    if (lane == 0) warp_part[wid] = __popc(m);
    __syncthreads();
    int off = 0;
#pragma unroll
    for (int w = 0; w < kTile / 32; ++w) off += w < wid ? warp_part[w] : 0;
    if (part) kjs[off + __popc(m & ((1u << lane) - 1u))] = kj;
    if (r == 0) {
      int tot = 0;
#pragma unroll
      for (int w = 0; w < kTile / 32; ++w) tot += warp_part[w];
      nchunk_part = tot;
    }
    __syncthreads();
    const int np = nchunk_part;
    // this CTA's tiles of the chunk: i = i0, i0 + kMaskSplit, ... (global
    // partial index ord + i congruent to blockIdx.y)
    const int g = static_cast<int>(blockIdx.y);
    const int i0 = ((g - ord) % kMaskSplit + kMaskSplit) % kMaskSplit;
    const int mine = np > i0 ? (np - i0 + kMaskSplit - 1) / kMaskSplit : 0;
    for (int b0 = 0; b0 < mine; b0 += kMaskBatch) {
      const int nb = min(kMaskBatch, mine - b0);
      if (b0 > 0) __syncthreads();  // the previous batch's bounds are no longer read
#pragma unroll
      for (int x = 0; x < kMaskBatch; ++x) {
        if (x < nb) {
          const int j = kjs[i0 + (b0 + x) * kMaskSplit] * kTile + r;
          sb[x][r] = j < Skv ? make_int4(__ldg(lts + bbase + j), __ldg(lte + bbase + j),
                                         __ldg(uts + bbase + j), __ldg(ute + bbase + j))
                             : make_int4(0, 0x7fffffff, 0, 0);
        }
      }
      __syncthreads();
      for (int x = 0; x < nb; ++x) {
        uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int c = 0; c < kTile; ++c) {
          const int4 v = sb[x][c];
          const bool hid = (v.x <= R && R < v.y) || (v.z <= R && R < v.w);
          w[c >> 5] |= (hid ? 1u : 0u) << (c & 31);
        }
        const int i = i0 + (b0 + x) * kMaskSplit;
        masks[(static_cast<size_t>(first + ord + i) * kTile + r)] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
    ord += np;
  }
}

// One warp per (bh, q-tile pair p): the union of the non-empty k-tiles of
// q-tiles 2p and 2p+1 (the second absent when nQ is odd), ascending, each
// entry (kj << 4) | (class_a << 2) | class_b, a non-empty ragged last k-tile
// as PARTIAL; info = {entries, tiles of 2p, tiles of 2p+1, their sum}.  The
// classes come from the block summary by the same rule as the table's, so
// the pairs need not wait for the rows' pass.
__device__ __forceinline__ void classify_pair(int w, const int32_t* __restrict__ summary, int nBH,
                                              int nQ, int nK, int nP, int Sq, int Skv,
                                              int4* pair_info, int32_t* pair_list) {
  const int lane = threadIdx.x & 31;
  if (w >= nBH * nP) return;
  const int bh = w / nP, p = w - bh * nP;
  const int32_t* sm = summary + static_cast<size_t>(bh) * nK * 8;
  const int ra0 = 2 * p * kTile, ra1 = min(ra0 + kTile, Sq);
  const bool has_b = 2 * p + 1 < nQ;
  const int rb0 = ra0 + kTile, rb1 = min(rb0 + kTile, Sq);
  int32_t* lst = pair_list + static_cast<size_t>(w) * nK;
  const unsigned lt_mask = (1u << lane) - 1u;
  const bool ragged = (Skv & (kTile - 1)) != 0;
  int cnt = 0, na = 0, nb = 0;
  for (int base = 0; base < nK; base += 32) {
    const int kj = base + lane;
    int ca = CLS_EMPTY, cb = CLS_EMPTY;
    if (kj < nK) {
      int s[8];
      load_summary(sm + kj * 8, s);
      ca = classify(s, ra0, ra1);
      cb = has_b ? classify(s, rb0, rb1) : CLS_EMPTY;
      if (ragged && kj == nK - 1) {
        if (ca != CLS_EMPTY) ca = CLS_PARTIAL;
        if (cb != CLS_EMPTY) cb = CLS_PARTIAL;
      }
    }
    const bool any = ca != CLS_EMPTY || cb != CLS_EMPTY;
    const unsigned m = __ballot_sync(0xffffffffu, any);
    if (any) lst[cnt + __popc(m & lt_mask)] = (kj << 4) | (ca << 2) | cb;
    cnt += __popc(m);
    na += __popc(__ballot_sync(0xffffffffu, ca != CLS_EMPTY));
    nb += __popc(__ballot_sync(0xffffffffu, cb != CLS_EMPTY));
  }
  if (lane == 0) pair_info[w] = make_int4(cnt, na, nb, na + nb);
}

// One warp per (bh, k-tile): the ascending list of non-empty q-tiles.
__device__ __forceinline__ void classify_col(int w, const int32_t* __restrict__ summary, int nBH,
                                             int nQ, int nK, int Sq, int32_t* col_count,
                                             int32_t* col_list) {
  const int lane = threadIdx.x & 31;
  if (w >= nBH * nK) return;
  int s[8];
  load_summary(summary + static_cast<size_t>(w) * 8, s);
  int32_t* lst = col_list + static_cast<size_t>(w) * nQ;
  const unsigned lt_mask = (1u << lane) - 1u;
  int cnt = 0;
  for (int base = 0; base < nQ; base += 32) {
    const int qi = base + lane;
    int cls = CLS_EMPTY;
    if (qi < nQ) {
      const int r0 = qi * kTile;
      cls = classify(s, r0, min(r0 + kTile, Sq));  // the rows' pass writes the table
    }
    const unsigned m = __ballot_sync(0xffffffffu, cls != CLS_EMPTY);
    if (cls != CLS_EMPTY) lst[cnt + __popc(m & lt_mask)] = (qi << 2) | cls;
    cnt += __popc(m);
  }
  if (lane == 0) col_count[w] = cnt;
}

// Rows, columns and the forward's pairs in one launch (all read only the
// block summary): blocks [0, row_blocks) classify q-tile rows, the next
// col_blocks k-tile columns, the rest q-tile pairs.  Eight warps per block,
// one row, column or pair each.
__global__ void __launch_bounds__(256) classify_kernel(
    const int32_t* __restrict__ summary, int nBH, int nQ, int nK, int nP, int Sq, int Skv,
    uint8_t* table, int32_t* row_count, int32_t* row_list, int32_t* row_mask,
    unsigned long long* slot_counter, int mask_cap, int row_blocks, int col_blocks,
    int32_t* col_count, int32_t* col_list, int4* pair_info, int32_t* pair_list) {
  const int wib = threadIdx.x >> 5;
  const int blk = static_cast<int>(blockIdx.x);
  if (blk < row_blocks)
    classify_row(blk * 8 + wib, summary, nBH, nQ, nK, Sq, Skv, table, row_count, row_list,
                 row_mask, slot_counter, mask_cap);
  else if (blk < row_blocks + col_blocks)
    classify_col((blk - row_blocks) * 8 + wib, summary, nBH, nQ, nK, Sq, col_count, col_list);
  else
    classify_pair((blk - row_blocks - col_blocks) * 8 + wib, summary, nBH, nQ, nK, nP, Sq, Skv,
                  pair_info, pair_list);
}

// ------------------------------------------------------------------ order
// Unit order: (b, h) ascending; within one (b, h) the nT units t by cost
// counts[b][hm][t] in [0, maxc] descending, ties by t ascending (longest
// first).  One CTA per (b, h): histogram, scan in descending cost, stable
// scatter by one warp in t order.
// One block per (b, unit head h); Hu = H / G unit heads.  G > 1: the units
// belong to K/V heads, each shared by query heads h*G .. h*G+G-1, and a
// unit's cost is the sum of their counts (maxc covers the sum).
// Up to three orders are built by one launch: blocks [0, jobs[0].blocks)
// make the first, the next jobs[1].blocks the second, and so on.
struct OrderJob {
  const int32_t* counts;
  int stride, G, nT, maxc, blocks;
  int32_t* order;
};
struct OrderJobs {
  OrderJob job[3];
  int n;
};

__global__ void __launch_bounds__(256) order_kernel(const __grid_constant__ OrderJobs J, int H,
                                                    int Hm) {
  int bh = blockIdx.x, ji = 0;
  while (ji + 1 < J.n && bh >= J.job[ji].blocks) {
    bh -= J.job[ji].blocks;
    ++ji;
  }
  const int32_t* __restrict__ counts = J.job[ji].counts;
  const int stride = J.job[ji].stride, G = J.job[ji].G, nT = J.job[ji].nT, maxc = J.job[ji].maxc;
  int32_t* order = J.job[ji].order;
  extern __shared__ int sh[];
  int* hist = sh;             // maxc + 1
  int* cst = sh + maxc + 1;   // nT costs of this (b, h)
  __shared__ int wsum[8];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Hu = H / G;
  const int b = bh / Hu, h = bh - b * Hu;
  for (int i = tid; i <= maxc; i += blockDim.x) hist[i] = 0;
  for (int t = tid; t < nT; t += blockDim.x) {
    int c = 0;
    for (int j = 0; j < G; ++j) {
      const int hm = Hm == 1 ? 0 : h * G + j;
      c += counts[(static_cast<size_t>(b * Hm + hm) * nT + t) * stride];
    }
    cst[t] = c;
  }
  __syncthreads();
  for (int t = tid; t < nT; t += blockDim.x) atomicAdd(&hist[cst[t]], 1);
  __syncthreads();
  // exclusive scan over r = maxc - c (descending cost), each thread a segment
  const int n = maxc + 1;
  const int seg = (n + blockDim.x - 1) / blockDim.x;
  const int r_lo = min(n, tid * seg), r_hi = min(n, r_lo + seg);
  int local = 0;
  for (int r = r_lo; r < r_hi; ++r) local += hist[maxc - r];
  int incl = local;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    int x = lane < nw ? wsum[lane] : 0;
    int xi = x;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, xi, off);
      if (lane >= off) xi += y;
    }
    if (lane < nw) wsum[lane] = xi - x;  // exclusive prefix of warp totals
  }
  __syncthreads();
  int run = wsum[warp] + incl - local;
  for (int r = r_lo; r < r_hi; ++r) {
    const int c = maxc - r;
    const int hc = hist[c];
    hist[c] = run;
    run += hc;
  }
  __syncthreads();
  if (warp == 0) {
    const unsigned lt_mask = (1u << lane) - 1u;
    int32_t* out = order + static_cast<size_t>(bh) * nT;
    for (int t0 = 0; t0 < nT; t0 += 32) {
      const int t = t0 + lane;
      const bool valid = t < nT;
      const int c = valid ? cst[t] : -1;
      const unsigned peers = __match_any_sync(0xffffffffu, c);
      int base = 0;
      if (valid) {
        base = hist[c];
        out[base + __popc(peers & lt_mask)] = bh * nT + t;
      }
      __syncwarp();
      if (valid && lane == __ffs(peers) - 1) hist[c] = base + __popc(peers);
      __syncwarp();
    }
  }
}

// ------------------------------------------------------------------ varlen
// Bounds of a packed batch: key j of sequence [a, b) (a = cu[s] <= j < b =
// cu[s+1]) is seen by rows [j, b) (causal) or [a, b): lower interval
// [b, total), upper interval [0, j) or [0, a).  The sequence is found by a
// binary search over cu[0..n].  Thread 0..n also checks that cu is a
// partition of [0, total) (cu[0] = 0, non-decreasing, cu[n] = total) and
// otherwise sets *bad; keys outside every sequence (only possible then) get
// bounds that hide them from every row.
__global__ void varlen_bounds_kernel(const int32_t* __restrict__ cu, int n, int total, int causal,
                                     int32_t* __restrict__ out, int* bad) {
  const int stride = gridDim.x * blockDim.x;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i <= n; i += stride) {
    const int c = cu[i];
    const bool ok = (i == 0 ? c == 0 : c >= cu[i - 1]) && (i < n || c == total) && c <= total;
    if (!ok && bad) atomicOr(bad, 1);
  }
  for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < total; j += stride) {
    int lo = 0, hi = n;  // find the last s in [0, n) with cu[s] <= j
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (cu[mid] <= j) lo = mid; else hi = mid;
    }
    const int a = cu[lo], b = cu[lo + 1];
    int4 v;
    if (a <= j && j < b) v = make_int4(b, total, 0, causal ? j : a);
    else v = make_int4(0, total, 0, 0);  // hidden from every row
    out[j] = v.x;
    out[total + j] = v.y;
    out[2 * total + j] = v.z;
    out[3 * total + j] = v.w;
  }
}

cudaError_t launch_varlen_bounds(const int32_t* cu, int n, int total, int causal, int32_t* out,
                                 int* bad, cudaStream_t s) {
  const int want = (total + 255) / 256;
  varlen_bounds_kernel<<<want < 1024 ? (want < 1 ? 1 : want) : 1024, 256, 0, s>>>(cu, n, total,
                                                                                 causal, out, bad);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ localize
__global__ void localize_kernel(const int32_t* __restrict__ in, int32_t* __restrict__ out,
                                long long n, const __grid_constant__ ChunkMap cm) {
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int x = in[i];
    int best = 0;
    for (int c = 0; c < cm.n; ++c) {
      if (cm.start[c] <= x) best = max(best, cm.offset[c] + min(x - cm.start[c], cm.len[c]));
    }
    out[i] = best;
  }
}

// ------------------------------------------------------------------ launchers
cudaError_t launch_summary(const Plan& p, const int32_t* lts, const int32_t* lte,
                           const int32_t* uts, const int32_t* ute, char* ws, cudaStream_t s) {
  dim3 grid(p.nK, p.B * p.Hm);
  prof_begin(K_SUMMARY, s);
  summary_kernel<<<grid, kTile, 0, s>>>(lts, lte, uts, ute, p.Sq, p.Skv, p.nK,
                                        reinterpret_cast<int32_t*>(ws + p.L.summary),
                                        reinterpret_cast<int*>(ws + p.L.status));
  prof_end(K_SUMMARY, s);
  return cudaGetLastError();
}

cudaError_t launch_classify(const Plan& p, char* ws, int mode, cudaStream_t s) {
  const int nBH = p.B * p.Hm;
  const int32_t* summ = reinterpret_cast<const int32_t*>(ws + p.L.summary);
  uint8_t* table = reinterpret_cast<uint8_t*>(ws + p.L.table);
  // q-tile rows (with their mask slots: the dQ pass walks them and the
  // forward's tile masks are filed by them), for the backward k-tile
  // columns, for the forward q-tile pairs
  const int row_blocks = ceil_div(nBH * p.nQ, 8);
  const int col_blocks = mode != FM_WS_FWD ? ceil_div(nBH * p.nK, 8) : 0;
  const int pair_blocks = mode != FM_WS_BWD ? ceil_div(nBH * p.nP, 8) : 0;
  prof_begin(K_CLASSIFY, s);
  classify_kernel<<<row_blocks + col_blocks + pair_blocks, 256, 0, s>>>(
      summ, nBH, p.nQ, p.nK, p.nP, p.Sq, p.Skv, table, reinterpret_cast<int32_t*>(ws + p.L.row_count),
      reinterpret_cast<int32_t*>(ws + p.L.row_list), reinterpret_cast<int32_t*>(ws + p.L.row_mask),
      reinterpret_cast<unsigned long long*>(ws + p.L.status + 8), p.mask_cap, row_blocks, col_blocks,
      reinterpret_cast<int32_t*>(ws + p.L.col_count), reinterpret_cast<int32_t*>(ws + p.L.col_list),
      reinterpret_cast<int4*>(ws + p.L.pair_info), reinterpret_cast<int32_t*>(ws + p.L.pair_list));
  prof_end(K_CLASSIFY, s);
  return cudaGetLastError();
}

cudaError_t launch_tile_masks(const Plan& p, const int32_t* lts, const int32_t* lte,
                              const int32_t* uts, const int32_t* ute, char* ws, cudaStream_t s) {
  prof_begin(K_TILE_MASKS, s);
  tile_mask_kernel<<<dim3(p.B * p.Hm * p.nQ, kMaskSplit), kTile, 0, s>>>(
      lts, lte, uts, ute, p.nQ, p.nK, p.Skv, reinterpret_cast<const int32_t*>(ws + p.L.row_count),
      reinterpret_cast<const int32_t*>(ws + p.L.row_list),
      reinterpret_cast<const int32_t*>(ws + p.L.row_mask), reinterpret_cast<uint4*>(ws + p.L.masks));
  prof_end(K_TILE_MASKS, s);
  return cudaGetLastError();
}

cudaError_t launch_orders(const Plan& p, char* ws, unsigned which, cudaStream_t s) {
  // forward: q-tile pairs, cost = the non-empty tiles of both rows
  // (pair_info[.][3]); dK/dV: k-tile columns, dQ: q-tile rows, cost = their
  // non-empty tiles
  OrderJobs J{};
  size_t smem = 0;
  int blocks = 0;
  for (int which_one : {ORDER_PAIRS, ORDER_COLS, ORDER_ROWS}) {
    if (!(which & (1u << which_one))) continue;
    OrderJob& jb = J.job[J.n++];
    jb.stride = 1;
    jb.G = 1;
    if (which_one == ORDER_PAIRS) {
      jb.nT = p.nP; jb.maxc = 2 * p.nK; jb.stride = 4;
      jb.counts = reinterpret_cast<const int32_t*>(ws + p.L.pair_info) + 3;
      jb.order = reinterpret_cast<int32_t*>(ws + p.L.fwd_order);
    } else if (which_one == ORDER_COLS) {
      // dK/dV units belong to K/V heads: G query heads' columns each
      jb.nT = p.nK; jb.maxc = p.G * p.nQ; jb.G = p.G;
      jb.counts = reinterpret_cast<const int32_t*>(ws + p.L.col_count);
      jb.order = reinterpret_cast<int32_t*>(ws + p.L.bwd_order);
    } else {
      jb.nT = p.nQ; jb.maxc = p.nK;
      jb.counts = reinterpret_cast<const int32_t*>(ws + p.L.row_count);
      jb.order = reinterpret_cast<int32_t*>(ws + p.L.row_order);
    }
    jb.blocks = p.B * (p.H / jb.G);
    blocks += jb.blocks;
    const size_t need = static_cast<size_t>(jb.maxc + 1 + jb.nT) * 4;
    if (need > smem) smem = need;
  }
  if (J.n == 0) return cudaSuccess;
  const size_t limit = 200 * 1024;
  if (smem > limit) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(order_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(limit));
  if (e != cudaSuccess) return e;
  prof_begin(K_ORDER, s);
  order_kernel<<<blocks, 256, smem, s>>>(J, p.H, p.Hm);
  prof_end(K_ORDER, s);
  return cudaGetLastError();
}

cudaError_t launch_localize(const int32_t* in, int32_t* out, long long n_values,
                            const ChunkMap& cm, cudaStream_t s) {
  const long long want = (n_values + 255) / 256;
  const int grid = static_cast<int>(want < 4096 ? (want < 1 ? 1 : want) : 4096);
  prof_begin(K_LOCALIZE, s);
  localize_kernel<<<grid, 256, 0, s>>>(in, out, n_values, cm);
  prof_end(K_LOCALIZE, s);
  return cudaGetLastError();
}

}  // namespace fm
