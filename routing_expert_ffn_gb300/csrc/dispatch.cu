// Dispatch (histogram -> scan -> stable scatter -> row gather), Combine, and the
// m-tile tables the grouped GEMMs schedule from.
//
// Dispatch is the single-GPU form of the expert-parallel Dispatch all-to-all
// (FarSkip-Collective review, "The reading"; T_Dispatch in the ledger's Eq. 9):
// every routed (token, expert) pair gets a slot in an expert-contiguous
// buffer, tokens of one expert in ascending token order.  Combine is the
// single-GPU form of the Combine all-to-all plus the gated sum, the shared
// expert and the residual base (Eq. 6 with its o_0 term, referee minor 1).
//
// Two index paths give the same slots.  The one the ABI calls ranks pairs in
// parallel blocks of 1024 (warp match + popc, block prefix), scans the
// (expert, block) counts (inside the scatter's CTAs when the table is small,
// else in one CTA of its own), and scatters rows token by token.  The chunked
// path (per-chunk counts, scan over (expert, chunk), in-chunk ranks by one
// warp, slot-driven row gather) serves the no-workspace entry point.  Ranks come from a
// warp match + popc in pair order, so the permutation is the same on every
// run; the combine sums in a fixed order.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Per chunk of kDispatchChunk tokens: how many of its pairs go to each expert.
__global__ void __launch_bounds__(256)
    dispatch_hist_kernel(const int32_t* __restrict__ idx, int T, int E, int k, int n_chunks,
                         int32_t* __restrict__ chunk_counts, unsigned* status) {
  __shared__ int cnt[256];
  const int c = blockIdx.x;
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  const long long p0 = static_cast<long long>(c) * kDispatchChunk * k;
  const long long p1 = static_cast<long long>(min(T, (c + 1) * kDispatchChunk)) * k;
  for (long long p = p0 + threadIdx.x; p < p1; p += blockDim.x) {
    const int e = idx[p];
    if (e < 0 || e >= E) {
      record_status(status, MOE_ERR_DEVICE_INDEX);
      continue;
    }
    atomicAdd(&cnt[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    chunk_counts[static_cast<long long>(e) * n_chunks + c] = cnt[e];
}

// One CTA per chunk: all threads stage the chunk's expert ids in shared
// memory, then warp 0 walks the pairs in (token, j) order, 32 at a time; lanes
// holding the same expert get consecutive slots in lane order.
constexpr int kScatterThreads = 128;
__global__ void __launch_bounds__(kScatterThreads)
    dispatch_scatter_kernel(const int32_t* __restrict__ idx, int T, int E, int k, int n_chunks,
                            const int32_t* __restrict__ chunk_base, int32_t* __restrict__ perm,
                            int32_t* __restrict__ slot_of) {
  __shared__ int base[256];
  __shared__ int s_idx[kDispatchChunk * 32];  // k <= 32
  const int c = blockIdx.x;
  const long long p0 = static_cast<long long>(c) * kDispatchChunk * k;
  const long long p1 = static_cast<long long>(min(T, (c + 1) * kDispatchChunk)) * k;
  const int n = static_cast<int>(p1 - p0);
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    base[e] = chunk_base[static_cast<long long>(e) * n_chunks + c];
  for (int i = threadIdx.x; i < n; i += blockDim.x) s_idx[i] = idx[p0 + i];
  __syncthreads();
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  const unsigned lt = lanemask_lt();
  for (int ib = 0; ib < n; ib += 32) {
    const int i = ib + lane;
    const long long p = p0 + i;
    int e = -1;
    if (i < n) {
      e = s_idx[i];
      if (e < 0 || e >= E) e = -1;
    }
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0) {
      const int slot = base[e] + __popc(peers & lt);
      perm[slot] = static_cast<int32_t>(p / k);
      slot_of[p] = slot;
    } else if (i < n) {
      slot_of[p] = -1;  // out-of-range expert (flagged by the histogram): no slot
    }
    __syncwarp();
    if (e >= 0 && lane == 31 - __clz(peers)) base[e] += __popc(peers);
    __syncwarp();
  }
}

// Parallel stable ranks, three kernels:
//   dispatch_local_kernel: block b takes pairs [1024 b, 1024 b + 1024); each
//     pair's rank among the block's earlier pairs with the same expert (warp
//     match + popc, then a prefix over the block's 32 warps), and the block's
//     per-expert counts, stored expert-major in blk[e][b].
//   dispatch_block_scan_kernel: exclusive prefix of blk in expert-major order
//     (so expert e's slots start at offsets[e] and, inside e, block b's pairs
//     follow blocks < b), plus counts and offsets.
//   scatter_rows_kernel: slot = blk[e][b] + local rank; writes slot_of, perm and
//     the row x_perm[slot] = x[token].
constexpr int kLocalPairs = 1024;
__global__ void __launch_bounds__(kLocalPairs)
    dispatch_local_kernel(const int32_t* __restrict__ idx, int P, int E, int n_blk,
                          int32_t* __restrict__ local_rank, int32_t* __restrict__ blk,
                          unsigned* status) {
  extern __shared__ int wh_flat[];  // [kLocalPairs / 32][E]
  auto wh = [&](int w, int x) -> int& { return wh_flat[w * E + x]; };
  // The trigger follows the wait: the scatter after this kernel reads x before its own
  // wait, and x is complete once this kernel's wait has returned.
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < (kLocalPairs / 32) * E; i += blockDim.x) wh_flat[i] = 0;
  __syncthreads();
  const int p = blockIdx.x * kLocalPairs + threadIdx.x;
  int e = -1;
  if (p < P) {
    e = idx[p];
    if (e < 0 || e >= E) {
      record_status(status, MOE_ERR_DEVICE_INDEX);
      e = -1;
    }
  }
  const unsigned peers = __match_any_sync(0xffffffffu, e);
  const int r = __popc(peers & lanemask_lt());
  if (e >= 0 && lane == __ffs(peers) - 1) wh(warp, e) = __popc(peers);
  __syncthreads();
  for (int x = threadIdx.x; x < E; x += blockDim.x) {
    int run = 0;
    for (int w = 0; w < kLocalPairs / 32; ++w) {
      const int c = wh(w, x);
      wh(w, x) = run;
      run += c;
    }
    blk[static_cast<long long>(x) * n_blk + blockIdx.x] = run;
  }
  __syncthreads();
  if (p < P) local_rank[p] = e >= 0 ? wh(warp, e) + r : -1;
}

// One CTA: out <- exclusive prefix of the (expert, block) count table in (expert-major,
// so expert e's slots start at offsets[e] and inside e block b's pairs follow blocks < b),
// plus counts and offsets.  out may be in (each piece is read before it is written).
// The table goes through shared memory in coalesced pieces of kScanPiece entries, each
// scanned by block_scan_smem and offset by the total of the pieces before it.  An empty
// table (n_blk = 0) gives zeros.
constexpr int kScanPiece = 8192;
__device__ int block_scan_smem(int* a, int n, int* wsum);
__device__ __forceinline__ int pad32(int i);
__global__ void __launch_bounds__(1024)
    dispatch_block_scan_kernel(const int32_t* in, int32_t* out, int E, int n_blk,
                               int32_t* __restrict__ counts, int32_t* __restrict__ offsets) {
  __shared__ int piece[kScanPiece + kScanPiece / 32 + 1];  // padded (pad32)
  __shared__ int wsum[33];
  const long long N = static_cast<long long>(E) * n_blk;
  pdl_trigger();
  pdl_wait();
  int carry = 0;
  for (long long base = 0; base < N; base += kScanPiece) {
    const int n = static_cast<int>(min(static_cast<long long>(kScanPiece), N - base));
    for (int i = threadIdx.x; i < n; i += blockDim.x) piece[pad32(i)] = in[base + i];
    __syncthreads();
    const int total = block_scan_smem(piece, n, wsum);  // ends with a barrier
    for (int i = threadIdx.x; i < n; i += blockDim.x) out[base + i] = carry + piece[pad32(i)];
    carry += total;
    __syncthreads();  // the piece is rewritten by the next iteration
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    offsets[e] = n_blk > 0 ? out[static_cast<long long>(e) * n_blk] : 0;
  if (threadIdx.x == 0) offsets[E] = carry;
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) counts[e] = offsets[e + 1] - offsets[e];
}

// Shared-memory tables that block_scan_smem scans are stored padded: entry i at pad32(i),
// one spare word after every 32, so that threads reading consecutive segments of any
// length hit distinct banks (a segment of 32 per thread would otherwise put a whole warp
// on one bank).  A padded table of n entries takes pad32(n) + 1 words.
__device__ __forceinline__ int pad32(int i) { return i + (i >> 5); }

// Exclusive prefix of the padded table a[0..n) by the whole CTA (blockDim a multiple of 32,
// at most 1024); returns the total.  Each thread sums a contiguous segment, the segment
// sums are scanned across the warp (shuffles) and the warps (shared memory), and each
// thread rewrites its segment.
__device__ int block_scan_smem(int* a, int n, int* wsum /* 33 ints */) {
  const int nt = blockDim.x, t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int seg = (n + nt - 1) / nt;
  const int lo = min(n, t * seg), hi = min(n, lo + seg);
  int mine = 0;
  for (int i = lo; i < hi; ++i) mine += a[pad32(i)];
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int v = lane < (nt >> 5) ? wsum[lane] : 0;
    int wi = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    wsum[lane] = wi - v;
    if (lane == 31) wsum[32] = wi;
  }
  __syncthreads();
  int run = wsum[warp] + incl - mine;
  for (int i = lo; i < hi; ++i) {
    const int c = a[pad32(i)];
    a[pad32(i)] = run;
    run += c;
  }
  __syncthreads();
  return wsum[32];
}

// For every pair p: slot = base[e][p / kLocalPairs] + local_rank[p]; slot_of[p] = slot,
// perm[slot] = p / k, x_perm[slot] = x[p / k].  One warp per token: lane j < k
// resolves pair (t, j), the warp reads the token's row once (in chunks of
// kRowChunk 16-byte vectors per lane, held in registers) and writes it to each
// of the token's k slots.  A pair with an out-of-range expert gets slot_of -1
// and no row.
// SCAN: blk holds the raw (expert, block) counts; every CTA scans the table in
// shared memory (it is small: E x ceil(P / 1024) entries) and CTA 0 writes
// counts and offsets -- this replaces a separate scan launch.  Otherwise blk
// is already the exclusive prefix.
constexpr int kRowChunk = 8;
// Largest count table the scatter scans in shared memory (8.3 KB of dynamic shared memory:
// 4 bytes per entry, padded by one word in 32).  Larger tables take the one-CTA scan: every
// scatter CTA would otherwise re-read and re-scan a table that long (measured on the
// Qwen3-30B-A3B-shaped layer's 8192-entry table: 71.5 us fused, 60.5 us with the one-CTA scan).
// scatter_scan_limit() checks at set-up that this, plus the kernel's static shared memory and
// the dynamic region's alignment, fits what a launch may use without opting in.
constexpr int kScatterScanMaxEntries = 2048;
// STATS (bf16 rows, for the condensation that follows in the same layer call): the warp also
// forms the row's fp32 norm and 64-bit content hash while the row is in its registers, in the
// same element order and with the same arithmetic as the condensation's own row statistics, and
// writes them at each of the token's slots (and resets the slot's earliest-similar-row entry).
template <typename T, bool SCAN, bool STATS>
__global__ void __launch_bounds__(256)
    scatter_rows_kernel(const T* __restrict__ x, const int32_t* __restrict__ idx,
                        const int32_t* __restrict__ local_rank, const int32_t* __restrict__ blk,
                        int n_blk, int E, int T_tok, int k, int d, T* __restrict__ x_perm,
                        int32_t* __restrict__ perm, int32_t* __restrict__ slot_of,
                        int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                        RowStatsOut stats, int split, unsigned* status) {
  constexpr int V = Act<T>::kVec;
  const int nv = d / V;
  const int P = T_tok * k;
  extern __shared__ int tab[];
  __shared__ int wsum[33];
  pdl_trigger();
  // `split` warps share a token (1 with STATS), each moving one slice of its row to all of
  // its slots, so that small batches still have enough rows in flight
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int sub = gw % split;
  const int warps = ((gridDim.x * blockDim.x) >> 5) / split;
  const int nvs = (nv + split - 1) / split;
  const int vbeg = sub * nvs, vend = min(nv, vbeg + nvs);
  const int lane = threadIdx.x & 31;
  int t = gw / split;
  // The first token's row chunk is loaded before the programmatic-launch wait (x is
  // complete when this kernel starts: dispatch_local_kernel, the kernel before it, triggers
  // only after its own wait) and its routing right after, both before the table scan, so
  // their latency overlaps the previous kernel's tail and the scan; each later token's are
  // loaded at the end of the previous token's iteration.
  uint4 r[kRowChunk];
  int e = -1, lr = -1;
  auto load_row = [&](int tok) {
    const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<long long>(tok) * d);
#pragma unroll
    for (int u = 0; u < kRowChunk; ++u) {
      const int v = vbeg + u * 32 + lane;
      if (v < vend) r[u] = src[v];
    }
  };
  auto load_routing = [&](int tok) {
    e = -1;
    lr = -1;
    if (lane < k) {
      const int p = tok * k + lane;
      e = idx[p];
      lr = local_rank[p];
    }
  };
  auto load_token = [&](int tok) {
    load_row(tok);
    load_routing(tok);
  };
  if (t < T_tok) load_row(t);
  pdl_wait();
  if (t < T_tok) load_routing(t);
  if (SCAN) {
    const int N = E * n_blk;
    for (int i = threadIdx.x; i < N; i += blockDim.x) tab[pad32(i)] = blk[i];
    __syncthreads();
    const int total = block_scan_smem(tab, N, wsum);
    if (blockIdx.x == 0) {
      for (int ee = threadIdx.x; ee < E; ee += blockDim.x) {
        const int o = tab[pad32(ee * n_blk)];
        offsets[ee] = o;
        counts[ee] = (ee + 1 < E ? tab[pad32((ee + 1) * n_blk)] : total) - o;
      }
      if (threadIdx.x == 0) offsets[E] = total;
    }
  }
  for (; t < T_tok; t += warps) {
    const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<long long>(t) * d);
    int slot = -1;
    if (lane < k) {
      const int p = t * k + lane;
      if (e >= 0 && e < E && lr >= 0) {
        const int ti = e * n_blk + p / kLocalPairs;
        slot = (SCAN ? tab[pad32(ti)] : blk[ti]) + lr;
        if (slot >= P) {
          record_status(status, MOE_ERR_DEVICE_INDEX);
          slot = -1;
        }
      }
      if (sub == 0) {
        slot_of[p] = slot;
        if (slot >= 0) perm[slot] = t;
      }
    }
    float ss = 0.f;
    unsigned long long h = 0x9E3779B97F4A7C15ull * (lane + 1);
    for (int v0 = vbeg; v0 < vend; v0 += 32 * kRowChunk) {
      if (v0 > vbeg) {
#pragma unroll
        for (int u = 0; u < kRowChunk; ++u) {
          const int v = v0 + u * 32 + lane;
          if (v < vend) r[u] = src[v];
        }
      }
      if (STATS) {
#pragma unroll
        for (int u = 0; u < kRowChunk; ++u) {
          if (v0 + u * 32 + lane >= nv) break;
          const uint32_t w[4] = {r[u].x, r[u].y, r[u].z, r[u].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float lo = __uint_as_float(w[i] << 16), hi = __uint_as_float(w[i] & 0xFFFF0000u);
            ss = fmaf(lo, lo, ss);
            ss = fmaf(hi, hi, ss);
            h = (h ^ w[i]) * 0x100000001B3ull;
            h ^= h >> 29;
          }
        }
      }
      for (int j = 0; j < k; ++j) {
        const int s = __shfl_sync(0xffffffffu, slot, j);
        if (s < 0) continue;
        uint4* dst = reinterpret_cast<uint4*>(x_perm + static_cast<long long>(s) * d);
#pragma unroll
        for (int u = 0; u < kRowChunk; ++u) {
          const int v = v0 + u * 32 + lane;
          if (v < vend) dst[v] = r[u];
        }
      }
    }
    if (STATS) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        ss += __shfl_xor_sync(0xffffffffu, ss, off);
        h ^= __shfl_xor_sync(0xffffffffu, h, off) * 0xBF58476D1CE4E5B9ull;
      }
      // every lane holds the sum of squares; lane 0's hash is the row's
      const unsigned long long h0 = __shfl_sync(0xffffffffu, h, 0);
      if (lane < k && slot >= 0) {
        stats.norm[slot] = sqrtf(ss);
        stats.hash[slot] = h0;
        stats.first[slot] = kNoHit;
      }
    }
    if (t + warps < T_tok) load_token(t + warps);
  }
}

// dst[r] = src[rows[r]] for r < *n_rows_dev; one warp per row, 16-byte vectors.
template <typename T>
__global__ void __launch_bounds__(256)
    gather_rows_kernel(const T* __restrict__ src, const int32_t* __restrict__ rows,
                       const int* __restrict__ n_rows_dev, int src_rows, int d,
                       T* __restrict__ dst, unsigned* status) {
  constexpr int V = Act<T>::kVec;
  pdl_trigger();
  pdl_wait();
  const int n_rows = *n_rows_dev;
  const int nv = d / V;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  const int lane = threadIdx.x & 31;
  for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < n_rows; r += warps) {
    const int s = rows[r];
    if (s < 0 || s >= src_rows) {
      if (lane == 0) record_status(status, MOE_ERR_DEVICE_INDEX);
      continue;
    }
    const uint4* a = reinterpret_cast<const uint4*>(src + static_cast<long long>(s) * d);
    uint4* b = reinterpret_cast<uint4*>(dst + static_cast<long long>(r) * d);
    for (int v = lane; v < nv; v += 32) b[v] = a[v];
  }
}

// out[t] = r[t] + shared[t] + sum_j g[t,j] * y[rep(slot_of[t,j])], fp32 accumulate.
// partial (nullable): p[t] = r[t] + shared[t], the same fp32 sum before the
// routed terms, rounded once.
// One CTA per token, one 16-byte vector per thread (blockDim = d / V).  The loads that do
// not depend on the routing (residual base, shared output) are issued before the token's
// slots and gates are fetched, so the CTA pays one memory round trip before its routed-row
// loads instead of two.  inputs_ready: x and residual are complete before this kernel
// starts (the layer's own chain guarantees it: the kernel before this one triggers its
// dependents only after its own wait), so they are read before the programmatic-launch
// wait and overlap the previous kernel's tail.
template <typename T>
__global__ void __launch_bounds__(1024)
    combine_kernel(const T* __restrict__ y, const T* __restrict__ shared_out,
                   const int32_t* __restrict__ slot_of, const int32_t* __restrict__ rep_of,
                   const float* __restrict__ gate, const T* __restrict__ x,
                   const T* residual, int residual_mode, T* out, T* __restrict__ partial, int d,
                   int k, int P, int inputs_ready, unsigned* status) {
  constexpr int V = Act<T>::kVec;
  __shared__ long long s_row[32];
  __shared__ float s_g[32];
  const int t = blockIdx.x;
  const int v = threadIdx.x;  // this thread's 16-byte vector of the row
  const bool act = v < d / V;
  const long long rowoff = static_cast<long long>(t) * d + static_cast<long long>(v) * V;
  const bool use_x = residual_mode == MOE_RES_INPUT || residual_mode == MOE_RES_INPUT_PLUS_EXTERNAL;
  const bool use_r =
      residual_mode == MOE_RES_EXTERNAL || residual_mode == MOE_RES_INPUT_PLUS_EXTERNAL;
  float acc[V], tmp[V];
#pragma unroll
  for (int i = 0; i < V; ++i) acc[i] = 0.f;
  pdl_trigger();
  if (inputs_ready && act) {
    if (use_x) {
      load_vec_f32_cs<T>(x + rowoff, tmp);
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] += tmp[i];
    }
    if (use_r) {
      load_vec_f32_cs<T>(residual + rowoff, tmp);
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] += tmp[i];
    }
  }
  pdl_wait();
  if (!inputs_ready && act) {
    if (use_x) {
      load_vec_f32_cs<T>(x + rowoff, tmp);
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] += tmp[i];
    }
    if (use_r) {
      load_vec_f32_cs<T>(residual + rowoff, tmp);
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] += tmp[i];
    }
  }
  // the shared output's load is in flight while the slots are fetched
  uint4 sh = make_uint4(0u, 0u, 0u, 0u);
  if (shared_out && act) sh = __ldcs(reinterpret_cast<const uint4*>(shared_out + rowoff));
  if (threadIdx.x < k) {
    int s = slot_of[static_cast<long long>(t) * k + threadIdx.x];
    if (s >= 0 && s < P && rep_of) s = rep_of[s];
    float g = gate[static_cast<long long>(t) * k + threadIdx.x];
    if (s < 0 || s >= P) {
      record_status(status, MOE_ERR_DEVICE_INDEX);
      s = 0;  // read a valid row with weight 0: the loop below needs no branch
      g = 0.f;
    }
    s_row[threadIdx.x] = s;
    s_g[threadIdx.x] = g;
  }
  __syncthreads();
  if (!act) return;
  if (shared_out) {
    load_vec_f32<T>(reinterpret_cast<const T*>(&sh), tmp);
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] += tmp[i];
  }
  if (partial) store_vec_f32<T>(partial + rowoff, acc);
  // branch-free over the k routed rows (unrolled, so several row loads are in flight)
#pragma unroll 4
  for (int j = 0; j < k; ++j) {
    const float g = s_g[j];
    load_vec_f32_cs<T>(y + s_row[j] * d + static_cast<long long>(v) * V, tmp);
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = fmaf(g, tmp[i], acc[i]);
  }
  store_vec_f32_cs<T>(out + rowoff, acc);
}

__global__ void __launch_bounds__(256)
    build_mtiles_kernel(const int32_t* __restrict__ counts, const int32_t* __restrict__ offsets_in,
                        int fixed_rows, int n_groups,
                        int32_t* __restrict__ offsets_out, int4* __restrict__ mt_info,
                        int32_t* __restrict__ group_mt_begin) {
  __shared__ int s_rows[256];
  __shared__ int s_off[257];
  __shared__ int s_mt[257];
  pdl_trigger();
  pdl_wait();
  for (int g = threadIdx.x; g < n_groups; g += blockDim.x)
    s_rows[g] = counts ? counts[g] : offsets_in ? offsets_in[g + 1] - offsets_in[g] : fixed_rows;
  __syncthreads();
  if (threadIdx.x == 0) {
    int off = 0, mt = 0;
    for (int g = 0; g < n_groups; ++g) {
      s_off[g] = off;
      s_mt[g] = mt;
      off += s_rows[g];
      mt += (s_rows[g] + kMTile - 1) / kMTile;
    }
    s_off[n_groups] = off;
    s_mt[n_groups] = mt;
  }
  __syncthreads();
  for (int g = threadIdx.x; g <= n_groups; g += blockDim.x) {
    group_mt_begin[g] = s_mt[g];
    if (offsets_out) offsets_out[g] = s_off[g];
  }
  for (int g = threadIdx.x; g < n_groups; g += blockDim.x) {
    const int rows = s_rows[g];
    for (int i = 0; i * kMTile < rows; ++i)
      mt_info[s_mt[g] + i] = make_int4(g, s_off[g] + i * kMTile, min(kMTile, rows - i * kMTile), s_off[g]);
  }
}

}  // namespace

size_t dispatch_scratch_bytes(int T, int E) {
  const size_t n_chunks = static_cast<size_t>(ceil_div(T, kDispatchChunk));
  return 2 * n_chunks * static_cast<size_t>(E) * sizeof(int32_t);
}

cudaError_t launch_dispatch(int act_dtype, const void* x, const int32_t* topk_idx, int T, int d,
                            int E, int k, int32_t* counts, int32_t* offsets, int32_t* perm,
                            int32_t* slot_of, void* x_perm, void* scratch, unsigned* status,
                            cudaStream_t stream) {
  const int n_chunks = ceil_div(T, kDispatchChunk);
  int32_t* chunk_counts = static_cast<int32_t*>(scratch);
  int32_t* chunk_base = chunk_counts + static_cast<size_t>(n_chunks) * E;
  if (T > 0) {
    dispatch_hist_kernel<<<n_chunks, 256, 0, stream>>>(topk_idx, T, E, k, n_chunks, chunk_counts,
                                                       status);
  }
  dispatch_block_scan_kernel<<<1, 1024, 0, stream>>>(chunk_counts, chunk_base, E, n_chunks, counts,
                                                      offsets);
  if (T == 0) return cudaGetLastError();
  dispatch_scatter_kernel<<<n_chunks, kScatterThreads, 0, stream>>>(topk_idx, T, E, k, n_chunks, chunk_base,
                                                       perm, slot_of);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_gather_rows(act_dtype, x, T, perm, offsets + E, T * k, d, x_perm, status, stream);
}

size_t dispatch_auto_scratch_bytes(int T, int k, int E) {
  const size_t P = static_cast<size_t>(T) * k;
  const size_t n_blk = (P + kLocalPairs - 1) / kLocalPairs;
  return ((P * sizeof(int32_t) + 255) & ~size_t(255)) + n_blk * E * sizeof(int32_t);
}

namespace {
// Largest (expert, block) table the scatter scans in its own shared memory on the current
// device: kScatterScanMaxEntries, unless the scatter's static shared memory plus the
// alignment of the dynamic region leave less than that within the per-launch default
// (0: every table takes the one-CTA scan).
int scatter_scan_limit() {
  static OncePerDevice<64> once;
  static int limit[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  int lim = 0;
  const cudaError_t e = once.run(dev, [&]() -> cudaError_t {
    int per_block = 0;
    cudaError_t r = cudaDeviceGetAttribute(&per_block, cudaDevAttrMaxSharedMemoryPerBlock, dev);
    if (r != cudaSuccess) return r;
    cudaFuncAttributes fa_f, fa_b;
    cudaFuncAttributes fa_s;
    if ((r = cudaFuncGetAttributes(&fa_f, scatter_rows_kernel<float, true, false>)) != cudaSuccess)
      return r;
    if ((r = cudaFuncGetAttributes(&fa_b, scatter_rows_kernel<__nv_bfloat16, true, false>)) !=
        cudaSuccess)
      return r;
    if ((r = cudaFuncGetAttributes(&fa_s, scatter_rows_kernel<__nv_bfloat16, true, true>)) !=
        cudaSuccess)
      return r;
    size_t stat = fa_f.sharedSizeBytes > fa_b.sharedSizeBytes ? fa_f.sharedSizeBytes
                                                              : fa_b.sharedSizeBytes;
    if (fa_s.sharedSizeBytes > stat) stat = fa_s.sharedSizeBytes;
    // static bytes rounded up to 128, plus 128 bytes for the dynamic region's alignment
    const long long room = static_cast<long long>(per_block) -
                           static_cast<long long>((stat + 127) / 128 * 128) - 128;
    // a padded table of n entries takes n + n / 32 + 1 words
    const long long words = room > 0 ? room / static_cast<long long>(sizeof(int)) : 0;
    const long long fit = words > 1 ? (words - 1) * 32 / 33 : 0;
    lim = static_cast<int>(fit < kScatterScanMaxEntries ? fit : kScatterScanMaxEntries);
    if (dev < 64) limit[dev] = lim;
    return cudaSuccess;
  });
  if (e != cudaSuccess) return 0;
  return dev < 64 ? limit[dev] : lim;
}
}  // namespace

cudaError_t launch_dispatch_auto(int act_dtype, const void* x, const int32_t* topk_idx, int T,
                                 int d, int E, int k, int32_t* counts, int32_t* offsets,
                                 int32_t* perm, int32_t* slot_of, void* x_perm, void* scratch,
                                 int num_sms, unsigned* status, cudaStream_t stream,
                                 const RowStatsOut* stats) {
  const long long P = static_cast<long long>(T) * k;
  if (P == 0)
    return launch_dispatch(act_dtype, x, topk_idx, T, d, E, k, counts, offsets, perm, slot_of,
                           x_perm, scratch, status, stream);
  const int n_blk = static_cast<int>((P + kLocalPairs - 1) / kLocalPairs);
  int32_t* local_rank = static_cast<int32_t*>(scratch);
  int32_t* blk = reinterpret_cast<int32_t*>(static_cast<char*>(scratch) +
                                            ((P * sizeof(int32_t) + 255) & ~size_t(255)));
  cudaError_t err = launch_pdl(dispatch_local_kernel, dim3(n_blk), dim3(kLocalPairs),
                               sizeof(int) * (kLocalPairs / 32) * E, stream, topk_idx,
                               static_cast<int>(P), E, n_blk, local_rank, blk, status);
  if (err != cudaSuccess) return err;
  const long long table = static_cast<long long>(E) * n_blk;
  const bool scan_in_smem = table <= scatter_scan_limit();
  if (!scan_in_smem) {
    err = launch_pdl(dispatch_block_scan_kernel, dim3(1), dim3(1024), 0, stream,
                     static_cast<const int32_t*>(blk), blk, E, n_blk, counts, offsets);
    if (err != cudaSuccess) return err;
  }
  // warps per token: small batches (fewer than 16 tokens per SM) share each row among up to
  // 8 warps, each slice at least two 16-byte vectors per lane (the row statistics need whole
  // rows).  Measured: the 64-token decode scatter 12.1 -> 10.0 us; two warps per token on the
  // 4096-token DeepSeek-V2-Lite layer changed nothing (its stores are bandwidth-bound).
  const int nv = d / (act_dtype == MOE_F32 ? 4 : 8);
  int split = 1;
  while (stats == nullptr && split < 8 && static_cast<long long>(T) * split < 16ll * num_sms &&
         nv >= 64 * split)
    split *= 2;
  const long long want = (static_cast<long long>(T) * split + 7) / 8;  // 8 warps per block
  const int blocks = static_cast<int>(want < 8ll * num_sms ? want : 8ll * num_sms);
  const size_t smem = scan_in_smem ? sizeof(int) * (table + table / 32 + 1) : 0;
  if (act_dtype == MOE_F32) {
    const float* xf = static_cast<const float*>(x);
    float* xp = static_cast<float*>(x_perm);
    err = scan_in_smem ? launch_pdl(scatter_rows_kernel<float, true, false>, dim3(blocks),
                                    dim3(256), smem, stream, xf, topk_idx, local_rank, blk, n_blk,
                                    E, T, k, d, xp, perm, slot_of, counts, offsets, RowStatsOut{},
                                    split, status)
                       : launch_pdl(scatter_rows_kernel<float, false, false>, dim3(blocks),
                                    dim3(256), 0, stream, xf, topk_idx, local_rank, blk, n_blk, E,
                                    T, k, d, xp, perm, slot_of, counts, offsets, RowStatsOut{},
                                    split, status);
  } else {
    const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
    __nv_bfloat16* xp = static_cast<__nv_bfloat16*>(x_perm);
    const bool st = stats != nullptr;
    auto kern = scan_in_smem ? (st ? scatter_rows_kernel<__nv_bfloat16, true, true>
                                   : scatter_rows_kernel<__nv_bfloat16, true, false>)
                             : (st ? scatter_rows_kernel<__nv_bfloat16, false, true>
                                   : scatter_rows_kernel<__nv_bfloat16, false, false>);
    err = launch_pdl(kern, dim3(blocks), dim3(256), scan_in_smem ? smem : 0, stream, xb, topk_idx,
                     local_rank, blk, n_blk, E, T, k, d, xp, perm, slot_of, counts, offsets,
                     st ? *stats : RowStatsOut{}, split, status);
  }
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

cudaError_t launch_gather_rows(int act_dtype, const void* src, int src_rows, const int32_t* rows,
                               const int* n_rows_dev, int max_rows, int d, void* dst,
                               unsigned* status, cudaStream_t stream) {
  if (max_rows <= 0) return cudaSuccess;
  const int blocks = min(ceil_div(max_rows, 8), 4096);
  const cudaError_t e =
      act_dtype == MOE_F32
          ? launch_pdl(gather_rows_kernel<float>, dim3(blocks), dim3(256), 0, stream,
                       static_cast<const float*>(src), rows, n_rows_dev, src_rows, d,
                       static_cast<float*>(dst), status)
          : launch_pdl(gather_rows_kernel<__nv_bfloat16>, dim3(blocks), dim3(256), 0, stream,
                       static_cast<const __nv_bfloat16*>(src), rows, n_rows_dev, src_rows, d,
                       static_cast<__nv_bfloat16*>(dst), status);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_combine(int act_dtype, const void* y_perm, const void* shared_out,
                           const int32_t* slot_of, const int32_t* rep_of, const float* topk_gate,
                           const void* x, const void* residual, int residual_mode, void* out, int T,
                           int d, int k, int P, unsigned* status, cudaStream_t stream,
                           void* partial, bool inputs_ready) {
  if (T == 0) return cudaSuccess;
  const int vec = act_dtype == MOE_F32 ? 4 : 8;
  const int threads = min(1024, max(32, ceil_div(d / vec, 32) * 32));
  const int ready = inputs_ready ? 1 : 0;
  if (act_dtype == MOE_F32)
    return launch_pdl(combine_kernel<float>, dim3(T), dim3(threads), 0, stream,
                      static_cast<const float*>(y_perm), static_cast<const float*>(shared_out),
                      slot_of, rep_of, topk_gate, static_cast<const float*>(x),
                      static_cast<const float*>(residual), residual_mode,
                      static_cast<float*>(out), static_cast<float*>(partial), d, k, P, ready,
                      status);
  return launch_pdl(combine_kernel<__nv_bfloat16>, dim3(T), dim3(threads), 0, stream,
                    static_cast<const __nv_bfloat16*>(y_perm),
                    static_cast<const __nv_bfloat16*>(shared_out), slot_of, rep_of, topk_gate,
                    static_cast<const __nv_bfloat16*>(x),
                    static_cast<const __nv_bfloat16*>(residual), residual_mode,
                    static_cast<__nv_bfloat16*>(out), static_cast<__nv_bfloat16*>(partial), d, k,
                    P, ready, status);
}

cudaError_t launch_build_mtiles(const int32_t* counts, const int32_t* offsets_in, int fixed_rows,
                                int n_groups, int32_t* offsets_out, int4* mt_info,
                                int32_t* group_mt_begin, cudaStream_t stream) {
  return launch_pdl(build_mtiles_kernel, dim3(1), dim3(256), 0, stream, counts, offsets_in,
                    fixed_rows, n_groups, offsets_out, mt_info, group_mt_begin);
}

}  // namespace moe
