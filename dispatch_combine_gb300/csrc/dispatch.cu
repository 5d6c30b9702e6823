// dispatch.cu -- dispatch as a permutation into expert-contiguous rows.
//
// "第十五章：多节点大模型推理" section 3.4: dispatch sends each token's
// activation to the k experts it was routed to, combine brings the results
// back; section 4.3 counts n_e, the assignments of expert e.  On one GPU the
// all-to-all becomes a stable counting sort of the T*k assignments
// a = t*k + j by expert:
//   1. per-chunk histograms (shared-memory counters, any order is fine),
//   2. one scan over chunks and experts -> counts, offsets and every chunk's
//      first row per expert,
//   3. one warp per chunk walks its assignments in order; lanes with the same
//      expert are ranked with __match_any_sync, so each assignment's row is
//      offsets[e] + (assignments to e before it) -- stable and independent
//      of scheduling,
//   4. a row gather x_perm[p] = x[src_token[p]] with 16-byte vectors.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kCountThreads = 256;

__global__ void __launch_bounds__(kCountThreads)
    dispatch_count_kernel(const int32_t *__restrict__ ids, int64_t n, int E, int chunk,
                          int32_t *__restrict__ chunk_counts, uint32_t *status) {
  pdl_begin();
  extern __shared__ int hist[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int64_t a0 = (int64_t)blockIdx.x * chunk;
  for (int q = threadIdx.x; q < chunk; q += blockDim.x) {
    const int64_t a = a0 + q;
    if (a < n) {
      const int id = ids[a];
      if (id >= 0 && id < E)
        atomicAdd(&hist[id], 1);
      else
        set_status(status, kStatusBadId);
    }
  }
  __syncthreads();
  int32_t *dst = chunk_counts + (size_t)blockIdx.x * E;
  for (int e = threadIdx.x; e < E; e += blockDim.x) dst[e] = hist[e];
}

// exclusive scan of one int per thread over a 1024-thread block;
// *total receives the sum of all 1024 values.
__device__ int block_exclusive_scan(int v, int *total) {
  __shared__ int warp_excl[32];
  __shared__ int grand;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) warp_excl[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int w = warp_excl[lane];
    int wi = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, wi, off);
      if (lane >= off) wi += o;
    }
    warp_excl[lane] = wi - w;
    if (lane == 31) grand = wi;
  }
  __syncthreads();
  const int res = warp_excl[warp] + incl - v;
  *total = grand;
  __syncthreads();  // the shared words may be reused by the next call
  return res;
}

// One CTA of 1024 threads (E <= 1024).  The chunks of expert e are split in
// Q consecutive ranges, Q = 1024 / (E rounded up to a power of two); thread
// (q, e) sums range q, the range sums are scanned in shared memory, then
// every thread rewrites its range as exclusive running counts.
__global__ void __launch_bounds__(1024)
    dispatch_scan_kernel(int32_t *__restrict__ chunk_counts, int nchunks, int E,
                         int32_t *__restrict__ counts, int32_t *__restrict__ offsets,
                         int32_t *__restrict__ mtile_base, int tile_rows, CapacityArgs cap,
                         uint32_t *__restrict__ zero_flags) {
  pdl_begin();
  // the down GEMM's split flags start every launch sequence at zero
  if (zero_flags)
    for (int i = threadIdx.x; i < kPairSplitFlagWords; i += blockDim.x) zero_flags[i] = 0;
  __shared__ int part[1024];
  int ep = 1;
  while (ep < E) ep <<= 1;
  // ranges per expert: enough to keep each range short, no more
  const int Q = min(1024 / ep, max(1, nchunks / 8));
  const int eq = threadIdx.x % ep, q = threadIdx.x / ep;
  const int per = (nchunks + Q - 1) / Q;
  const int c0 = q * per, c1 = min(nchunks, c0 + per);
  int local = 0;
  if (eq < E) {
    // sixteen loads in flight at a time (a range is up to a few hundred chunks)
    for (int c = c0; c < c1; c += 16) {
      int v[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) v[u] = (c + u < c1) ? chunk_counts[(size_t)(c + u) * E + eq] : 0;
#pragma unroll
      for (int u = 0; u < 16; ++u) local += v[u];
    }
  }
  part[threadIdx.x] = local;
  __syncthreads();
  int base = 0, run = 0;
  for (int q2 = 0; q2 < Q; ++q2) {
    const int v = part[q2 * ep + eq];
    if (q2 < q) base += v;
    run += v;
  }
  if (eq < E) {
    int r = base;
    for (int c = c0; c < c1; c += 16) {
      int v[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) v[u] = (c + u < c1) ? chunk_counts[(size_t)(c + u) * E + eq] : 0;
#pragma unroll
      for (int u = 0; u < 16; ++u)
        if (c + u < c1) {
          chunk_counts[(size_t)(c + u) * E + eq] = r;
          r += v[u];
        }
    }
  }
  // thread e < E (range q == 0 of expert e) carries expert e's total
  const int e = threadIdx.x;
  if (e >= E) run = 0;
  int total = 0;
  const int excl = block_exclusive_scan(e < E ? run : 0, &total);
  if (e < E) {
    counts[e] = run;
    offsets[e] = excl;
  }
  if (e == 0) offsets[E] = total;
  if (cap.kept) {
    // capacity: the first C rows of an expert stay, the rest overflow
    const int kept = (e < E) ? min(run, cap.capacity) : 0;
    int ovf_total = 0;
    const int ovf_excl = block_exclusive_scan((e < E) ? run - kept : 0, &ovf_total);
    if (e < E) {
      cap.kept[e] = kept;
      cap.ovf_offsets[e] = ovf_excl;
    }
    if (e == 0) cap.ovf_offsets[E] = ovf_total;
  }
  if (mtile_base) {
    int mt_total = 0;
    const int mt = (e < E) ? (run + tile_rows - 1) / tile_rows : 0;
    const int mt_excl = block_exclusive_scan(mt, &mt_total);
    if (e < E) mtile_base[e] = mt_excl;
    if (e == 0) mtile_base[E] = mt_total;
  }
}

constexpr int kScatterWarps = 4;

__global__ void __launch_bounds__(kScatterWarps * 32)
    dispatch_scatter_kernel(const int32_t *__restrict__ ids, int64_t n, int k, int E, int chunk,
                            int64_t nchunks, const int32_t *__restrict__ chunk_base,
                            const int32_t *__restrict__ offsets, int32_t *__restrict__ dest,
                            int32_t *__restrict__ src_token, CapacityArgs cap) {
  pdl_begin();
  extern __shared__ int cursor_all[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t ci = (int64_t)blockIdx.x * kScatterWarps + warp;
  if (ci >= nchunks) return;
  int *cursor = cursor_all + warp * E;
  for (int e = lane; e < E; e += 32) cursor[e] = chunk_base[ci * E + e] + offsets[e];
  __syncwarp();
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int s = 0; s < chunk / 32; ++s) {
    const int64_t a = ci * chunk + s * 32 + lane;
    int id = (a < n) ? ids[a] : -1;
    const bool valid = id >= 0 && id < E;
    if (!valid) id = -1;
    const unsigned grp = __match_any_sync(0xffffffffu, id);
    const int leader = __ffs(grp) - 1;
    const int rank = __popc(grp & lt_mask);
    int base = 0;
    if (valid && lane == leader) {
      base = cursor[id];
      cursor[id] = base + __popc(grp);
    }
    base = __shfl_sync(0xffffffffu, base, leader);
    __syncwarp();
    if (valid) {
      int p = base + rank;
      if (cap.kept) {
        // rank r inside the expert: padded row e*C + r, or an overflow row
        // (second round) after all padded rows, or none (drop)
        const int r = p - offsets[id];
        if (r < cap.capacity)
          p = id * cap.capacity + r;
        else if (cap.policy == MOE_OVERFLOW_SECOND_ROUND)
          p = E * cap.capacity + cap.ovf_offsets[id] + (r - cap.capacity);
        else
          p = -1;
      }
      dest[a] = p;
      if (p >= 0) src_token[p] = static_cast<int32_t>(a / k);
    }
  }
}

constexpr int kGatherWarps = 8;

__global__ void __launch_bounds__(kGatherWarps * 32)
    dispatch_gather_kernel(const uint4 *__restrict__ x, const int32_t *__restrict__ ids,
                           const int32_t *__restrict__ dest, int T, int k, int E,
                           const int32_t *__restrict__ offsets_end, int64_t n, int vec_per_row,
                           uint4 *__restrict__ x_perm, CapacityArgs cap) {
  pdl_begin();
  // Token-major: warp item (t, s) reads 4 KB segment s of x[t] once and
  // writes it to the rows dest[t*k + j] of the token's valid assignments, so
  // x is read once however many experts a token has.  Valid rows are
  // [0, offsets[E]) (with a capacity: the E*C padded rows, then the
  // overflow rows); assignments with an invalid id or no row (dropped) are
  // skipped, and rows without an assignment are left untouched.
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t pad = cap.kept ? static_cast<int64_t>(cap.E) * cap.capacity : 0;
  const int64_t rows = cap.kept ? pad + cap.ovf_offsets[cap.E]
                                : min(n, static_cast<int64_t>(*offsets_end));
  const int segs = (vec_per_row + 255) / 256;
  const int64_t items = static_cast<int64_t>(T) * segs;
  for (int64_t it = (int64_t)blockIdx.x * kGatherWarps + warp; it < items;
       it += (int64_t)gridDim.x * kGatherWarps) {
    const int t = static_cast<int>(it / segs);
    const int v0 = static_cast<int>(it - static_cast<int64_t>(t) * segs) * 256;
    int p = -1;
    if (lane < k) {
      const int64_t a = static_cast<int64_t>(t) * k + lane;
      const int id = ids[a];
      if (id >= 0 && id < E) {
        const int q = dest[a];
        if (q >= 0 && q < rows) p = q;
      }
    }
    const uint4 *src = x + (size_t)t * vec_per_row;
    uint4 r[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int v = v0 + u * 32 + lane;
      if (v < vec_per_row) r[u] = __ldg(src + v);
    }
    for (int j = 0; j < k; ++j) {
      const int pj = __shfl_sync(0xffffffffu, p, j);
      if (pj < 0) continue;
      uint4 *dst = x_perm + (size_t)pj * vec_per_row;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int v = v0 + u * 32 + lane;
        if (v < vec_per_row) dst[v] = r[u];
      }
    }
  }
}

// per-row fp32 block scales follow their row: dst[p, b] = src[src_token[p], b]
__global__ void __launch_bounds__(256)
    gather_scales_kernel(const float *__restrict__ src, const int32_t *__restrict__ src_token,
                         const int32_t *__restrict__ offsets_end, int64_t n, int T, int per_row,
                         float *__restrict__ dst) {
  pdl_begin();
  const int64_t rows = min(n, static_cast<int64_t>(*offsets_end));
  const int64_t total = rows * per_row;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t row = i / per_row;
    const int t = src_token[row];
    if (t < 0 || t >= T) continue;
    dst[i] = src[static_cast<int64_t>(t) * per_row + (i - row * per_row)];
  }
}

// mtile_base from offsets (layout 0) or masked_m clamped to M_max (layout 1)
__global__ void __launch_bounds__(1024)
    ffn_tiles_kernel(const int32_t *__restrict__ seg, const int32_t *__restrict__ seg2,
                     int layout, int E, int M_max, int tile_rows,
                     int32_t *__restrict__ mtile_base, uint32_t *status,
                     uint32_t *__restrict__ zero_flags) {
  pdl_begin();
  // the down GEMM's split flags start every launch sequence at zero
  if (zero_flags)
    for (int i = threadIdx.x; i < kPairSplitFlagWords; i += blockDim.x) zero_flags[i] = 0;
  const int e = threadIdx.x;
  int rows = 0, tiles2 = 0;
  if (e < E) {
    if (layout == kLayoutTwoSeg) {
      // the slab's rows (clamped to M_max), then the overflow rows
      rows = min(max(seg[e], 0), M_max);
      if (seg[e] > M_max || seg[e] < 0) set_status(status, kStatusOverflow);
      int r2 = seg2[e + 1] - seg2[e];
      if (r2 < 0) {
        set_status(status, kStatusBadId);
        r2 = 0;
      }
      tiles2 = (r2 + tile_rows - 1) / tile_rows;
    } else if (layout == MOE_LAYOUT_CONTIGUOUS) {
      rows = seg[e + 1] - seg[e];
      if (rows < 0) {
        set_status(status, kStatusBadId);
        rows = 0;
      }
    } else {
      rows = seg[e];
      if (rows > M_max) {
        set_status(status, kStatusOverflow);
        rows = M_max;
      }
      if (rows < 0) {
        set_status(status, kStatusBadId);
        rows = 0;
      }
    }
  }
  int total = 0;
  const int excl = block_exclusive_scan((rows + tile_rows - 1) / tile_rows + tiles2, &total);
  if (e < E) mtile_base[e] = excl;
  if (e == 0) mtile_base[E] = total;
}

// ---------------------------------------------------------------------------
// Dispatch onto physical expert copies ("ep-deploy" page, section "EPLB 与路由
// 约束": hot experts get copies; "第十五章" section 4.3: each assignment goes
// to one of its expert's equivalent copies, the less loaded one).  The
// logical dispatch runs first (its dest gives every assignment its stable
// rank r among its expert's assignments); the r-th assignment of expert e
// goes to copy r mod n_rep(e), the copies taken in slot order -- the least
// loaded copy at every step, ties to the first.  Rows are contiguous per
// physical slot, in slot order, stable in a = t*k + j inside a slot.
// ---------------------------------------------------------------------------

// One CTA of 1024 threads.  Warp 0 ranks the slots of each expert in
// increasing slot order (32 slots at a time, like the scatter): slot_rank[p]
// = the copy index of slot p, n_rep[e] = copies of e.  Then rep_first =
// exclusive scan of n_rep, rep_slots[rep_first[e] + i] = the i-th slot of e,
// counts_phys[p] = the assignments r < n_e with r mod n_rep == i, and
// offsets_phys = their exclusive scan in slot order.
__global__ void __launch_bounds__(1024)
    replica_plan_kernel(const int32_t *__restrict__ phys_expert, int P, int E,
                        const int32_t *__restrict__ counts_log, int32_t *__restrict__ n_rep,
                        int32_t *__restrict__ rep_first, int32_t *__restrict__ rep_slots,
                        int32_t *__restrict__ slot_rank, int32_t *__restrict__ counts_phys,
                        int32_t *__restrict__ offsets_phys, uint32_t *status) {
  pdl_begin();
  extern __shared__ int cursor[];  // [E]
  const int tid = threadIdx.x, lane = tid & 31;
  for (int e = tid; e < E; e += 1024) cursor[e] = 0;
  __syncthreads();
  if (tid < 32) {
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int p0 = 0; p0 < P; p0 += 32) {
      const int p = p0 + lane;
      int e = (p < P) ? phys_expert[p] : -1;
      if (p < P && (e < 0 || e >= E)) {
        set_status(status, kStatusBadId);
        e = -1;
      }
      const unsigned grp = __match_any_sync(0xffffffffu, e);
      const int leader = __ffs(grp) - 1;
      int base = 0;
      if (e >= 0 && lane == leader) {
        base = cursor[e];
        cursor[e] = base + __popc(grp);
      }
      base = __shfl_sync(0xffffffffu, base, leader);
      __syncwarp();
      if (p < P) slot_rank[p] = (e >= 0) ? base + __popc(grp & lt_mask) : -1;
    }
  }
  __syncthreads();
  // copies per expert and where each expert's copies start in rep_slots
  const int nr = (tid < E) ? cursor[tid] : 0;
  if (tid < E) {
    n_rep[tid] = nr;
    if (nr == 0 && counts_log[tid] > 0) set_status(status, kStatusBadId);  // routed, no copy
  }
  int total = 0;
  const int first = block_exclusive_scan(nr, &total);
  if (tid < E) rep_first[tid] = first;
  if (tid == 0) rep_first[E] = total;
  __syncthreads();  // rep_first visible (global, same block)
  // slot lists and per-slot counts, then their scan in slot order
  int carry = 0;
  for (int p0 = 0; p0 < P; p0 += 1024) {
    const int p = p0 + tid;
    int c = 0;
    if (p < P) {
      const int e = phys_expert[p];
      const int i = slot_rank[p];
      if (e >= 0 && e < E && i >= 0) {
        rep_slots[rep_first[e] + i] = p;
        const int ne = counts_log[e], m = n_rep[e];
        c = (ne > i) ? (ne - i + m - 1) / m : 0;
      }
      counts_phys[p] = c;
    }
    int chunk_total = 0;
    const int excl = block_exclusive_scan(c, &chunk_total);
    if (p < P) offsets_phys[p] = carry + excl;
    carry += chunk_total;
    __syncthreads();  // the scan's shared totals are reused by the next chunk
  }
  if (tid == 0) offsets_phys[P] = carry;
}

// dest / src_token of the physical rows: the r-th assignment of e goes to
// copy r mod n_rep(e), row offsets_phys[slot] + r / n_rep(e)
__global__ void __launch_bounds__(256)
    replica_scatter_kernel(const int32_t *__restrict__ ids, int64_t n, int k, int E,
                           const int32_t *__restrict__ offsets_log,
                           const int32_t *__restrict__ dest_log,
                           const int32_t *__restrict__ n_rep, const int32_t *__restrict__ rep_first,
                           const int32_t *__restrict__ rep_slots,
                           const int32_t *__restrict__ offsets_phys, int32_t *__restrict__ dest,
                           int32_t *__restrict__ src_token) {
  pdl_begin();
  for (int64_t a = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; a < n;
       a += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int e = ids[a];
    int row = -1;
    if (e >= 0 && e < E && n_rep[e] > 0) {
      const int m = n_rep[e];
      const int r = dest_log[a] - offsets_log[e];
      const int p = rep_slots[rep_first[e] + r % m];
      row = offsets_phys[p] + r / m;
      src_token[row] = static_cast<int32_t>(a / k);
    }
    dest[a] = row;
  }
}

}  // namespace

cudaError_t launch_dispatch_replicated(const int32_t *ids, int T, int k, int E, const void *x,
                                       int d, int P, const int32_t *phys_expert,
                                       int32_t *counts_phys, int32_t *offsets_phys,
                                       int32_t *src_token, int32_t *dest, void *x_perm,
                                       const ReplicaScratch &w, uint32_t *status,
                                       cudaStream_t s) {
  const int64_t n = static_cast<int64_t>(T) * k;
  if (n == 0) return cudaSuccess;
  // the logical dispatch: counts, offsets and each assignment's stable rank
  cudaError_t err = launch_dispatch(ids, T, k, E, nullptr, d, w.counts_log, w.offsets_log,
                                    w.src_log, w.dest_log, nullptr, w.chunk, w.mtile, 128,
                                    status, s);
  if (err != cudaSuccess) return err;
  MOE_LAUNCH_PDL(replica_plan_kernel, 1, 1024, E * sizeof(int), s, phys_expert, P, E,
                 static_cast<const int32_t *>(w.counts_log), w.n_rep, w.rep_first, w.rep_slots,
                 w.slot_rank, counts_phys, offsets_phys, status);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  const int64_t want = (n + 255) / 256;
  const int64_t cap = static_cast<int64_t>(num_sms()) * 8;
  MOE_LAUNCH_PDL(replica_scatter_kernel, static_cast<unsigned>(want < cap ? want : cap), 256, 0,
                 s, ids, n, k, E, static_cast<const int32_t *>(w.offsets_log),
                 static_cast<const int32_t *>(w.dest_log), static_cast<const int32_t *>(w.n_rep),
                 static_cast<const int32_t *>(w.rep_first),
                 static_cast<const int32_t *>(w.rep_slots),
                 static_cast<const int32_t *>(offsets_phys), dest, src_token);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  if (x != nullptr && x_perm != nullptr) {
    const int vec = d / 8;
    const int64_t items = static_cast<int64_t>(T) * ((vec + 255) / 256);
    const int64_t gwant = (items + kGatherWarps - 1) / kGatherWarps;
    const unsigned gblocks = static_cast<unsigned>(gwant < cap ? gwant : cap);
    MOE_LAUNCH_PDL(dispatch_gather_kernel, gblocks, kGatherWarps * 32, 0, s,
                   static_cast<const uint4 *>(x), ids, static_cast<const int32_t *>(dest), T, k,
                   E, static_cast<const int32_t *>(offsets_phys + P), n, vec,
                   static_cast<uint4 *>(x_perm), CapacityArgs{0, 0, 0, nullptr, nullptr});
    err = cudaGetLastError();
  }
  return err;
}

cudaError_t launch_dispatch(const int32_t *ids, int T, int k, int E, const void *x, int d,
                            int32_t *counts, int32_t *offsets, int32_t *src_token,
                            int32_t *dest, void *x_perm, int32_t *chunk_scratch,
                            int32_t *mtile_base, int tile_rows, uint32_t *status,
                            cudaStream_t s, CapacityArgs cap, uint32_t *zero_flags) {
  cap.E = E;
  const int64_t n = (int64_t)T * k;
  const int64_t nchunks = dispatch_num_chunks(n);
  const int chunk = dispatch_chunk(n);
  if (n == 0) return cudaSuccess;
  MOE_LAUNCH_PDL(dispatch_count_kernel, (unsigned)nchunks, kCountThreads, E * sizeof(int), s, 
      ids, n, E, chunk, chunk_scratch, status);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  MOE_LAUNCH_PDL(dispatch_scan_kernel, 1, 1024, 0, s, chunk_scratch, (int)nchunks, E, counts, offsets,
                                          mtile_base, tile_rows, cap, zero_flags);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const unsigned sblocks = (unsigned)((nchunks + kScatterWarps - 1) / kScatterWarps);
  MOE_LAUNCH_PDL(dispatch_scatter_kernel, sblocks, kScatterWarps * 32, kScatterWarps * E * sizeof(int), s, 
      ids, n, k, E, chunk, nchunks, chunk_scratch, offsets, dest, src_token, cap);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  if (x != nullptr && x_perm != nullptr) {
    const int vec = d / 8;
    const int64_t items = static_cast<int64_t>(T) * ((vec + 255) / 256);
    const int64_t want = (items + kGatherWarps - 1) / kGatherWarps;
    const int64_t grid_cap = (int64_t)num_sms() * 8;
    const unsigned gblocks = (unsigned)(want < grid_cap ? want : grid_cap);
    MOE_LAUNCH_PDL(dispatch_gather_kernel, gblocks, kGatherWarps * 32, 0, s, 
        static_cast<const uint4 *>(x), ids, dest, T, k, E, offsets + E, n, vec,
        static_cast<uint4 *>(x_perm), cap);
    err = cudaGetLastError();
  }
  return err;
}

cudaError_t launch_gather_rows(const void *src, int row_bytes, const float *src_scale,
                               int scales_per_row, const int32_t *ids, const int32_t *dest,
                               int k, int E, const int32_t *src_token,
                               const int32_t *offsets_end, int64_t n, int T, void *dst,
                               float *dst_scale, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const int vec = row_bytes / 16;
  const int64_t items = static_cast<int64_t>(T) * ((vec + 255) / 256);
  const int64_t want = (items + kGatherWarps - 1) / kGatherWarps;
  const int64_t grid_cap = (int64_t)num_sms() * 8;
  MOE_LAUNCH_PDL(dispatch_gather_kernel, (unsigned)(want < grid_cap ? want : grid_cap), kGatherWarps * 32, 0,
                           s, static_cast<const uint4 *>(src), ids, dest, T, k, E,
                                offsets_end, n, vec, static_cast<uint4 *>(dst),
                                CapacityArgs{0, 0, 0, nullptr, nullptr});
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess || !src_scale) return err;
  const int64_t scale_items = n * scales_per_row;
  const int64_t blocks = (scale_items + 255) / 256;
  MOE_LAUNCH_PDL(gather_scales_kernel, (unsigned)(blocks < grid_cap ? blocks : grid_cap), 256, 0, s, 
      src_scale, src_token, offsets_end, n, T, scales_per_row, dst_scale);
  return cudaGetLastError();
}

cudaError_t launch_ffn_tiles(const int32_t *seg, int layout, int E, int M_max, int tile_rows,
                             int32_t *mtile_base, uint32_t *status, cudaStream_t s,
                             const int32_t *seg2, uint32_t *zero_flags) {
  if (layout == kLayoutTwoSeg && seg2 == nullptr) return cudaErrorInvalidValue;
  MOE_LAUNCH_PDL(ffn_tiles_kernel, 1, 1024, 0, s, seg, seg2, layout, E, M_max, tile_rows,
                 mtile_base, status, zero_flags);
  return cudaGetLastError();
}

}  // namespace moe
