// Luffy token condensation inside each expert bucket (bf16 rows).
//
// Luffy review, "What carries the argument": only tokens routed to the same
// expert are compared (expert activation), similar tokens form groups in a
// token graph, one representative per group is sent and computed, and its
// expert output is reused by the group; referee major comment 1: a condensed
// token's forward uses its representative's output.  Reading taken here:
// walk a bucket in slot order keeping the set R of representatives; slot j is
// condensed onto the earliest r in R with cos(x_j, x_r) >= tau, else it joins R.
//
// Work split:
//   1. row_stats:   per dispatched row, fp32 L2 norm and a 64-bit content hash (inside a
//                   condensing layer the dispatch forms them instead).
//   2. tile list:   per bucket, the lower-triangle tiles (256 rows x 256 columns, a
//                   pair of the bucket's m-tiles) of its Gram matrix.
//   3. sim tiles:   tcgen05 GEMM of the bucket against itself on CTA pairs; the
//                   epilogue writes bits A[i][j] = (cos >= tau) for j < i (identical
//                   rows count as cos = 1; a zero row is otherwise dissimilar) and
//                   lowers each row's earliest similar row.
//   4. resolve:     rows with no similar row, or whose earliest similar row has none
//                   before it, are decided at once (a warp per 32 rows, all buckets).
//   5. greedy scan: one CTA per bucket that still has undecided rows walks the rows in
//                   order with R as a bitset; j's candidates are A[j] & R, its
//                   representative the lowest.  Rows go 32 at a time, one per lane: a
//                   row's lowest candidate among the representatives chosen before its
//                   group is its answer (they all precede the group's own); only rows
//                   with none are resolved in order against the group's new
//                   representatives, on one 32-bit word.  Fifteen warps search a
//                   group's older words while the group before it is being resolved.
// The decision cos >= tau is taken in fp32.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kScanThreads = 512;     // warp 0 resolves groups, the other warps stage and search ahead
constexpr int kScanHelpers = kScanThreads / 32 - 1;
constexpr int kMaxBucketRows = 65536;
constexpr int kMaxWords = kMaxBucketRows / 32;
constexpr int kScanBufWords = 12288;  // one of two staging buffers (48 KB)

// 4-byte asynchronous global -> shared copy (no register round trip: every copy
// a thread issues is in flight at once), and the wait for all of a thread's copies.
__device__ __forceinline__ void cp_async4(unsigned* dst, const unsigned* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// Per dispatched row: fp32 norm and a 64-bit content hash (a filter for identical rows,
// which are then compared element by element); resets the row's earliest-similar-row
// entry.  One warp per row; a lane's vectors are loaded kStatBatch at a time, so their
// loads are in flight together.
constexpr int kStatBatch = 4;
__global__ void __launch_bounds__(256)
    row_stats_kernel(const __nv_bfloat16* __restrict__ rows, const int32_t* __restrict__ offsets,
                     int E, int d, float* __restrict__ norm, unsigned long long* __restrict__ hash,
                     int32_t* __restrict__ first) {
  pdl_trigger();
  pdl_wait();
  const int n_rows = offsets[E];
  const int warps = (gridDim.x * blockDim.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int nv = d / 8;
  for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < n_rows; r += warps) {
    const uint4* p = reinterpret_cast<const uint4*>(rows + static_cast<long long>(r) * d);
    float ss = 0.f;
    unsigned long long h = 0x9E3779B97F4A7C15ull * (lane + 1);
    for (int v0 = 0; v0 < nv; v0 += 32 * kStatBatch) {
      uint4 q[kStatBatch];
#pragma unroll
      for (int u = 0; u < kStatBatch; ++u) {
        const int v = v0 + u * 32 + lane;
        q[u] = v < nv ? p[v] : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < kStatBatch; ++u) {
        if (v0 + u * 32 + lane >= nv) break;
        const uint32_t w[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
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
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      ss += __shfl_xor_sync(0xffffffffu, ss, off);
      h ^= __shfl_xor_sync(0xffffffffu, h, off) * 0xBF58476D1CE4E5B9ull;
    }
    // Every lane holds the full sum of squares; lane 0's hash depends on every lane's
    // words.  Lane 0 writes.
    if (lane == 0) {
      norm[r] = sqrtf(ss);
      hash[r] = h;
      first[r] = kNoHit;  // lowered by the similarity tiles
    }
  }
}

// Tile list of the lower triangle of every bucket's Gram matrix, and the
// start word of each bucket's bit matrix (rows of ceil(n_e / 32) words).  A tile is
// 256 rows (a pair of the bucket's m-tiles, run on a CTA pair) by 256 columns:
// {first m-tile, column tile | (1 << 16) when the bucket holds the pair's second m-tile}.
// The scratch is sized for buckets of at most max_rows rows (a bucket holds each token at
// most once).  A bucket longer than that (offsets from a routing that names one expert twice
// for a token) sets *overflow, flags MOE_ERR_DEVICE_INDEX, lists no tile, invalidates the
// history record being written (hist_header, nullable) and leaves every slot its own
// representative (greedy_scan reads *overflow).
__global__ void __launch_bounds__(256)
    sim_tiles_kernel(const int4* __restrict__ mt_info, const int32_t* __restrict__ group_mt_begin,
                     const int32_t* __restrict__ offsets, int E, int max_rows,
                     int2* __restrict__ tile_list, int32_t* __restrict__ n_list,
                     long long* __restrict__ bits_base, int32_t* __restrict__ overflow,
                     int32_t* __restrict__ hist_header, int32_t* __restrict__ unresolved,
                     int32_t* __restrict__ nrep_fast, int32_t* __restrict__ done,
                     unsigned* status) {
  __shared__ int s_cnt[1024];
  __shared__ int s_beg[1025];
  __shared__ int s_second[1024];
  __shared__ int s_over;
  pdl_trigger();
  pdl_wait();
  // the counts the resolve pass and the walk add up
  for (int e = threadIdx.x; e < E; e += blockDim.x) unresolved[e] = nrep_fast[e] = 0;
  if (threadIdx.x == 0) {
    *done = 0;
    s_over = 0;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int n = offsets[e + 1] - offsets[e];
    if (n < 0 || n > max_rows) s_over = 1;
  }
  __syncthreads();
  if (s_over) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) bits_base[e] = 0;
    if (threadIdx.x == 0) {
      *overflow = 1;
      *n_list = 0;
      if (hist_header) hist_header[0] = 0;
      record_status(status, MOE_ERR_DEVICE_INDEX);
    }
    return;
  }
  if (threadIdx.x == 0) *overflow = 0;
  const int n_mt = group_mt_begin[E];
  // Chunks of 1024 m-tiles; the running tile count carries across chunks.
  __shared__ int s_carry;
  if (threadIdx.x == 0) s_carry = 0;
  __syncthreads();
  for (int c0 = 0; c0 < n_mt; c0 += 1024) {
    for (int i = threadIdx.x; i < 1024; i += blockDim.x) {
      const int m = c0 + i;
      int cnt = 0, second = 0;
      if (m < n_mt) {
        const int4 t = mt_info[m];
        const int mb = group_mt_begin[t.x], me = group_mt_begin[t.x + 1];
        if (((m - mb) & 1) == 0) {  // the first m-tile of a pair
          second = m + 1 < me ? 1 : 0;
          const int4 u = second ? mt_info[m + 1] : t;
          const int li_end = u.y - u.w + u.z;  // one past the last local row of the pair
          cnt = (li_end + kTcTileN - 1) / kTcTileN;
        }
      }
      s_cnt[i] = cnt;
      s_second[i] = second;
    }
    __syncthreads();
    {
      // exclusive scan of the 1024 counts: 4 consecutive entries per thread, then the
      // threads' sums across each warp (shuffles) and across the warps (shared memory)
      __shared__ int s_wsum[32];
      const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
      const int per = 1024 / blockDim.x;  // 4 with 256 threads
      const int i0 = threadIdx.x * per;
      int mine = 0;
      for (int q = 0; q < per; ++q) mine += s_cnt[i0 + q];
      int incl = mine;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (lane == 31) s_wsum[warp] = incl;
      __syncthreads();
      int before = s_carry;
      for (int w = 0; w < warp; ++w) before += s_wsum[w];
      int run = before + incl - mine;
      for (int q = 0; q < per; ++q) {
        s_beg[i0 + q] = run;
        run += s_cnt[i0 + q];
      }
      if (threadIdx.x == blockDim.x - 1) s_beg[1024] = run;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 1024; i += blockDim.x) {
      for (int j = 0; j < s_cnt[i]; ++j)
        tile_list[s_beg[i] + j] = make_int2(c0 + i, j | (s_second[i] << 16));
    }
    __syncthreads();
    if (threadIdx.x == 0) s_carry = s_beg[1024];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    *n_list = s_carry;
    long long run = 0;
    for (int e = 0; e < E; ++e) {
      bits_base[e] = run;
      const long long n = offsets[e + 1] - offsets[e];
      run += n * ((n + 31) / 32);
    }
  }
}

// One CTA per bucket.  Warps 1-15 stage the bit rows of the next chunk of rows
// into one of two buffers (row pitch odd, so 32 rows at the same word offset sit
// in distinct banks) and search the current chunk's rows one 32-row group ahead
// of warp 0, which resolves the groups in order.
// Buckets whose 32-row group does not fit a buffer (more than 12256 rows) take
// the row-by-row walk over staged rows instead.
// Returns the bucket's representative count (in thread 0).
__device__ __forceinline__ int greedy_scan_bucket(
    const unsigned* __restrict__ bits, const long long* __restrict__ bits_base,
    const int32_t* __restrict__ offsets, const int32_t* __restrict__ overflow,
    const int32_t* __restrict__ unresolved, const int32_t* __restrict__ nrep_fast,
    int32_t* __restrict__ rep_of, unsigned* status) {
  extern __shared__ unsigned scan_smem[];
  unsigned* R = scan_smem;                  // kMaxWords: representatives so far, as a bitset
  unsigned* buf = scan_smem + kMaxWords;    // 2 x kScanBufWords
  const int e = blockIdx.x;
  const int off = offsets[e];
  const int n = offsets[e + 1] - off;
  const int W = (n + 31) >> 5;
  if (!*overflow && unresolved[e] == 0) {
    // resolve_kernel decided every row of the bucket
    return nrep_fast[e];
  }
  if (*overflow || n > kMaxBucketRows) {
    // no bit matrix: every slot is its own representative
    for (int i = threadIdx.x; i < n; i += blockDim.x) rep_of[off + i] = off + i;
    if (threadIdx.x == 0) record_status(status, MOE_ERR_DEVICE_INDEX);
    return max(n, 0);
  }
  for (int w = threadIdx.x; w < W; w += blockDim.x) R[w] = 0u;
  const unsigned* B = bits + bits_base[e];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pitch = W | 1;
  int reps = 0;
  if (32 * pitch <= kScanBufWords) {
    // Per 32-row group G (rows 32G .. 32G + 31 of the bucket) a row's lowest
    // candidate among the representatives chosen before the group lies in R's words
    // 0 .. G-1.  Words 0 .. G-2 are final once group G-2 is resolved, so the helper
    // warps search them one group ahead (an equal share of the words each, the lowest
    // hit per row merged by a shared-memory minimum) while warp 0 resolves group G-1;
    // warp 0 then checks only word G-1 for group G.
    __shared__ int best[2][32];  // per look-ahead group and row: lowest hit, INT_MAX for none
    if (threadIdx.x < 64) best[threadIdx.x >> 5][threadIdx.x & 31] = INT_MAX;
    const int rows_chunk = 32 * (kScanBufWords / (32 * pitch));
    const int n_chunks = (n + rows_chunk - 1) / rows_chunk;
    // rows [r0 + g0, r0 + g0 + cnt) of the chunk starting at row r0, into dst: row li
    // needs words 0 .. li / 32 only; the copies are asynchronous and waited for once,
    // before the chunk's last barrier
    auto stage_rows = [&](int r0, int g0, int cnt, unsigned* dst) {
      int rr = g0 + warp - 1;
      const unsigned* src = B + static_cast<long long>(r0 + rr) * W;
      unsigned* d = dst + rr * pitch;
      for (; rr < g0 + cnt; rr += kScanHelpers, src += kScanHelpers * W, d += kScanHelpers * pitch) {
        const int top = (r0 + rr) >> 5;
        for (int w = lane; w <= top; w += 32) cp_async4(d + w, src + w);
      }
    };
    if (warp != 0) {
      stage_rows(0, 0, min(rows_chunk, n), buf);
      cp_async_wait_all();
    }
    __syncthreads();
    for (int c = 0; c < n_chunks; ++c) {
      const unsigned* cur = buf + (c & 1) * kScanBufWords;
      const int r0 = c * rows_chunk;
      const int rows = min(rows_chunk, n - r0);
      const int ng = (rows + 31) >> 5;
      // the next chunk (there is one only after a full chunk, so it has at most ng
      // groups) is staged one group per iteration
      const int rows_next = c + 1 < n_chunks ? min(rows_chunk, n - r0 - rows_chunk) : 0;
      unsigned* nxt = buf + ((c + 1) & 1) * kScanBufWords;
      // iteration j: the helpers stage the next chunk's group j and search group j's
      // old words, warp 0 resolves group j - 1; every thread runs ng + 1 iterations and
      // one barrier in each
      for (int j = 0; j <= ng; ++j) {
        if (warp != 0) {
          if (32 * j < rows_next) stage_rows(r0 + rows_chunk, 32 * j, min(32, rows_next - 32 * j), nxt);
          if (j < ng) {
            const int g0 = 32 * j;
            const int G = (r0 + g0) >> 5;
            const int nw = max(G - 1, 0);
            const int h = warp - 1;
            const int wb = (h * nw) / kScanHelpers, we = ((h + 1) * nw) / kScanHelpers;
            int hit = -1;
            if (g0 + lane < rows) {
              const unsigned* row = cur + (g0 + lane) * pitch;
              // eight words per step: the loads of a step do not wait on each other
              for (int w = wb; w < we; w += 8) {
                unsigned m[8], any = 0u;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                  m[q] = (w + q < we) ? (row[w + q] & R[w + q]) : 0u;
                  any |= m[q];
                }
                if (any) {
                  int q = 7;
                  unsigned mq = m[7];
#pragma unroll
                  for (int u = 6; u >= 0; --u)
                    if (m[u]) q = u, mq = m[u];
                  hit = ((w + q) << 5) + __ffs(mq) - 1;
                  break;
                }
              }
            }
            if (hit >= 0) atomicMin(&best[j & 1][lane], hit);
          }
        } else if (j > 0) {
          const int g0 = 32 * (j - 1);
          const int i0 = r0 + g0;  // a multiple of 32: the group's columns are word G
          const int G = i0 >> 5;
          const int li = i0 + lane;
          const bool live = g0 + lane < rows;
          const unsigned* row = cur + (g0 + lane) * pitch;
          int old_hit = best[(j - 1) & 1][lane];
          best[(j - 1) & 1][lane] = INT_MAX;  // ready for group j + 1's search
          if (old_hit == INT_MAX) old_hit = -1;
          if (live && old_hit < 0 && G >= 1) {
            const unsigned m = row[G - 1] & R[G - 1];
            if (m) old_hit = ((G - 1) << 5) + __ffs(m) - 1;
          }
          // similarities to the group's earlier rows (A holds only columns below the row)
          const unsigned inw = live ? (row[G] & ((1u << lane) - 1u)) : 0u;
          const unsigned open = __ballot_sync(0xffffffffu, live && old_hit < 0);
          // an open row with no open row before it in its word is a new representative;
          // the others are decided in order against the representatives before them
          const unsigned dep = __ballot_sync(0xffffffffu, ((open >> lane) & 1u) && (inw & open));
          unsigned fresh = open & ~dep;
          for (unsigned dd = dep; dd; dd &= dd - 1u) {
            const int b = __ffs(dd) - 1;
            const unsigned wb = __shfl_sync(0xffffffffu, inw, b);
            if (!(wb & fresh)) fresh |= 1u << b;
          }
          if (live) {
            int rp;
            if (old_hit >= 0) rp = old_hit;
            else if ((fresh >> lane) & 1u) rp = li;
            else rp = i0 + __ffs(inw & fresh) - 1;
            rep_of[off + li] = off + rp;
          }
          reps += __popc(fresh);
          if (lane == 0) R[G] = fresh;
        }
        __syncthreads();
      }
      if (warp != 0) cp_async_wait_all();
      __syncthreads();
    }
  } else {
    // wide buckets: stage as many whole rows as fit both buffers, walk them one by one
    unsigned* stage = buf;
    const int stage_words = 2 * kScanBufWords;
    const int rows_per_chunk = max(1, stage_words / W);
    for (int r0 = 0; r0 < n; r0 += rows_per_chunk) {
      const int rows = min(rows_per_chunk, n - r0);
      __syncthreads();
      for (int i = threadIdx.x; i < rows * W; i += blockDim.x) {
        const int rr = i / W, w = i - rr * W;
        // only words strictly below the row's own index are meaningful
        stage[i] = (w * 32 < r0 + rr) ? B[static_cast<long long>(r0 + rr) * W + w] : 0u;
      }
      __syncthreads();
      if (warp == 0) {
        for (int rr = 0; rr < rows; ++rr) {
          const int li = r0 + rr;
          const int nw = (li + 31) >> 5;  // words holding columns < li
          int found = -1;
          for (int w0 = 0; w0 < nw && found < 0; w0 += 32) {
            const int w = w0 + lane;
            const unsigned cand = (w < nw) ? (stage[rr * W + w] & R[w]) : 0u;
            const unsigned hit = __ballot_sync(0xffffffffu, cand != 0u);
            if (hit) {
              const int src = __ffs(hit) - 1;
              const unsigned cw = __shfl_sync(0xffffffffu, cand, src);
              found = (w0 + src) * 32 + __ffs(cw) - 1;
            }
          }
          if (lane == 0) {
            if (found < 0) {
              R[li >> 5] |= 1u << (li & 31);
              rep_of[off + li] = off + li;
            } else {
              rep_of[off + li] = off + found;
            }
          }
          if (found < 0) ++reps;
          __syncwarp();
        }
      }
    }
  }
  return reps;
}

// One CTA per bucket (see greedy_scan_bucket).  The last CTA to finish also writes
// n_condensed = (number of slots) - (representatives of every bucket); *done counts the
// finished CTAs (zeroed by sim_tiles_kernel, reset here for the next call).
__global__ void __launch_bounds__(kScanThreads)
    greedy_scan_kernel(const unsigned* __restrict__ bits, const long long* __restrict__ bits_base,
                       const int32_t* __restrict__ offsets, const int32_t* __restrict__ overflow,
                       const int32_t* __restrict__ unresolved, const int32_t* __restrict__ nrep_fast,
                       int32_t* __restrict__ rep_of, int32_t* n_rep, int32_t* done,
                       int32_t* __restrict__ n_condensed, unsigned* status) {
  pdl_trigger();
  pdl_wait();
  const int reps =
      greedy_scan_bucket(bits, bits_base, offsets, overflow, unresolved, nrep_fast, rep_of, status);
  if (threadIdx.x == 0) {
    n_rep[blockIdx.x] = reps;
    __threadfence();
    if (atomicAdd(done, 1) == static_cast<int>(gridDim.x) - 1) {
      __threadfence();
      const volatile int32_t* nr = n_rep;
      int total = 0;
      for (int e = 0; e < static_cast<int>(gridDim.x); ++e) total += nr[e];
      *n_condensed = offsets[gridDim.x] - total;
      *done = 0;
    }
  }
}

// Rows decided without the walk.  For slot s (local row li of bucket e) let C be the rows
// before li that its bits mark similar.  first[s] = min C (local), or kNoHit when C is empty:
// the similarity GEMM's epilogue and the history lookup lower it with atomicMin as they write
// the bits.  resolve_kernel then decides two kinds of row exactly as the walk would: C empty ->
// a representative; m = min C with no similar row before it (m is then a representative, and
// the earliest candidate) -> condensed onto m.  Any other row is left to the walk: a bucket
// with such a row counts it in unresolved[e] and greedy_scan_kernel walks that bucket; the
// other buckets are complete (n_rep from nrep_fast).
__global__ void __launch_bounds__(256)
    resolve_kernel(const int32_t* __restrict__ first, const int32_t* __restrict__ offsets, int E,
                   const int32_t* __restrict__ overflow, int32_t* __restrict__ rep_of,
                   int32_t* __restrict__ unresolved, int32_t* __restrict__ nrep_fast) {
  __shared__ int off[257];
  pdl_trigger();
  pdl_wait();
  for (int i = threadIdx.x; i <= E; i += blockDim.x) off[i] = offsets[i];
  __syncthreads();
  if (*overflow) return;
  const int n_rows = off[E];
  const int lane = threadIdx.x & 31;
  const int stride = gridDim.x * blockDim.x;
  // warp-uniform trip count; the per-bucket counts are summed over the warp's lanes of one
  // bucket and added by one lane
  for (int base = blockIdx.x * blockDim.x + (threadIdx.x & ~31); base < n_rows; base += stride) {
    const int sl = base + lane;
    int lo = -1;
    bool is_rep = false, open = false;
    if (sl < n_rows) {
      lo = 0;
      int hi = E;
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (off[mid] <= sl) lo = mid; else hi = mid;
      }
      const int f = first[sl];
      if (f == kNoHit) {
        rep_of[sl] = sl;
        is_rep = true;
      } else if (first[off[lo] + f] == kNoHit) {
        rep_of[sl] = off[lo] + f;
      } else {
        open = true;
      }
    }
    const unsigned peers = __match_any_sync(0xffffffffu, lo);
    const int n_r = __popc(__ballot_sync(0xffffffffu, is_rep) & peers);
    const int n_o = __popc(__ballot_sync(0xffffffffu, open) & peers);
    if (lo >= 0 && lane == __ffs(peers) - 1) {
      if (n_r) atomicAdd(&nrep_fast[lo], n_r);
      if (n_o) atomicAdd(&unresolved[lo], n_o);
    }
  }
}

// tau > 1 or NaN: every slot is its own representative.
__global__ void identity_reps_kernel(const int32_t* offsets, int E, int P, int32_t* rep_of,
                                     int32_t* n_rep, int32_t* n_condensed) {
  const int n = offsets[E];
  for (int s = blockIdx.x * blockDim.x + threadIdx.x; s < n; s += gridDim.x * blockDim.x)
    rep_of[s] = s;
  if (blockIdx.x == 0) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) n_rep[e] = offsets[e + 1] - offsets[e];
    if (threadIdx.x == 0) *n_condensed = 0;
  }
  (void)P;
}

// One CTA per bucket: the bucket's representatives in slot order, at the bucket's own
// slots (rep_local[off_e + i] = slot of its i-th representative), and their count.  No CTA
// needs another bucket's count: gather_reps_kernel places the lists one after another.
__global__ void __launch_bounds__(1024)
    compact_reps_kernel(const int32_t* __restrict__ rep_of, const int32_t* __restrict__ offsets,
                        int E, int32_t* __restrict__ rep_local, int32_t* __restrict__ rep_counts) {
  __shared__ int s_warp[32];
  pdl_trigger();
  pdl_wait();
  const int e = blockIdx.x;
  const int off = offsets[e], n = offsets[e + 1] - off;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int base = 0;
  for (int c0 = 0; c0 < n; c0 += blockDim.x) {
    const int s = c0 + threadIdx.x;
    const bool is_rep = s < n && rep_of[off + s] == off + s;
    const unsigned b = __ballot_sync(0xffffffffu, is_rep);
    if (lane == 0) s_warp[warp] = __popc(b);
    __syncthreads();
    int before = 0, total = 0;
    for (int w = 0; w < 32; ++w) {
      if (w < warp) before += s_warp[w];
      total += s_warp[w];
    }
    if (is_rep) rep_local[off + base + before + __popc(b & ((1u << lane) - 1u))] = off + s;
    base += total;
    __syncthreads();
  }
  if (threadIdx.x == 0) rep_counts[e] = base;
}

// Row r of the compact representative list (r < rep_off[E], rep_off the exclusive prefix of
// the per-bucket counts): bucket e with rep_off[e] <= r < rep_off[e + 1], slot
// s = rep_local[offsets[e] + r - rep_off[e]]; writes rep_rows[r] = s and dst[r] = src[s].
// One warp per row, 16-byte vectors.
template <typename T>
__global__ void __launch_bounds__(256)
    gather_reps_kernel(const T* __restrict__ src, const int32_t* __restrict__ rep_local,
                       const int32_t* __restrict__ offsets, const int32_t* __restrict__ rep_off,
                       int E, int d, T* __restrict__ dst, int32_t* __restrict__ rep_rows) {
  constexpr int V = Act<T>::kVec;
  __shared__ int s_roff[257];
  __shared__ int s_off[257];
  pdl_trigger();
  pdl_wait();
  for (int i = threadIdx.x; i <= E; i += blockDim.x) {
    s_roff[i] = rep_off[i];
    s_off[i] = offsets[i];
  }
  __syncthreads();
  const int n_rows = s_roff[E];
  const int nv = d / V;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  const int lane = threadIdx.x & 31;
  for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < n_rows; r += warps) {
    int lo = 0, hi = E;  // s_roff[lo] <= r < s_roff[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_roff[mid] <= r) lo = mid; else hi = mid;
    }
    const int s = rep_local[s_off[lo] + r - s_roff[lo]];
    if (lane == 0) rep_rows[r] = s;
    const uint4* a = reinterpret_cast<const uint4*>(src + static_cast<long long>(s) * d);
    uint4* b = reinterpret_cast<uint4*>(dst + static_cast<long long>(r) * d);
    for (int v = lane; v < nv; v += 32) b[v] = a[v];
  }
}

// Expert (bucket) of a slot of the record: the largest e with off[e] <= s < off[e + 1];
// -1 if s is out of range.
__device__ __forceinline__ int bucket_of(const int* off, int E, int s) {
  if (s < 0 || s >= off[E]) return -1;
  int lo = 0, hi = E;  // off[lo] <= s < off[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (off[mid] <= s) lo = mid; else hi = mid;
  }
  return lo;
}

// Historical similarity: for every tile of the Gram tile list, each pair (li, lj), lj < li,
// of bucket e's slots takes the class its two tokens got at the previous call, found in the
// previous record's bucket that held both (their previous slots si > sj, both in it; a pair
// of tokens that shared two buckets got the same class in each).  Writes, in the bits layout
// of this call, the planes (the inherited classes) and the bits themselves (= the class; the
// similarity GEMM rewrites the bits of tiles with unclassified pairs), and lists the tiles
// with an unclassified pair for the GEMM.  One CTA per tile of up to 256 rows (grid-stride),
// 8 warps; a warp takes a row at a time.  A chunk of 32 columns whose tokens sat at consecutive slots of one
// previous bucket, with the row's token in that bucket too, is one 32-bit window of the
// previous row's planes (one lane, a funnel shift); any other chunk takes a lane per column,
// each searching its pair's previous buckets for a common one.
constexpr int kLookupThreads = 256;
constexpr int kLookupChunks = kTcTileN / 32;
__global__ void __launch_bounds__(kLookupThreads)
    hist_lookup_kernel(const int2* __restrict__ tile_list, const int32_t* __restrict__ n_list,
                       const int4* __restrict__ mt_info, const int32_t* __restrict__ offsets,
                       const int32_t* __restrict__ perm, int T, int k, int E,
                       const long long* __restrict__ bits_base, HistView prev,
                       uint2* __restrict__ planes_out, unsigned* __restrict__ bits,
                       int32_t* __restrict__ first, int2* __restrict__ cos_list,
                       int32_t* __restrict__ n_cos) {
  extern __shared__ int hsm[];
  int* poff = hsm;                      // [E + 1] previous offsets
  int* col_e = poff + (E + 1);          // [256][k] previous bucket of each column token's pairs
  int* col_s = col_e + kTcTileN * k;    // [256][k] and their slots
  int* row_e = col_s + kTcTileN * k;    // [256][k] the same for the tile's row tokens
  int* row_s = row_e + 2 * kMTile * k;  // [256][k]
  __shared__ int s_unknown;
  // per 32-column chunk: the previous bucket its tokens all held at consecutive slots from
  // s_ch_s0 (-1: none), so a row in that bucket reads its 32 classes without a search
  __shared__ int s_ch_e[kLookupChunks], s_ch_s0[kLookupChunks];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int P = T * k;
  const bool have = prev.header[0] == kHistMagic && prev.header[1] == T && prev.header[2] == k &&
                    prev.header[3] == E && prev.header[4] == P;
  if (have)
    for (int i = threadIdx.x; i <= E; i += blockDim.x) poff[i] = prev.offsets[i];
  const int n_tiles = *n_list;
  for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
    const int2 tl = tile_list[tile];
    const int4 m = mt_info[tl.x];
    // the pair's m-tiles are consecutive 128-row pieces of the bucket: rows row0 .. + nrows
    const int e = m.x, row0 = m.y, gbase = m.w;
    const int nrows = m.z + (((tl.y >> 16) & 1) ? mt_info[tl.x + 1].z : 0);
    const int n_e = offsets[e + 1] - offsets[e];
    const int W = (n_e + 31) >> 5;
    const int lj0 = (tl.y & 0xffff) * kTcTileN;
    const int li0 = row0 - gbase;
    if (threadIdx.x == 0) s_unknown = 0;
    __syncthreads();  // poff staged; the previous tile's reads of the tables are done
    if (have) {
      for (int q = threadIdx.x; q < kTcTileN * k; q += blockDim.x) {
        const int c = q / k, a = q - c * k;
        int pe = -1, ps = -1;
        if (lj0 + c < n_e) {
          const int tok = perm[gbase + lj0 + c];
          if (tok >= 0 && tok < T) {
            ps = prev.slot_of[static_cast<long long>(tok) * k + a];
            pe = bucket_of(poff, E, ps);
          }
        }
        col_e[q] = pe;
        col_s[q] = ps;
      }
      for (int q = threadIdx.x; q < 2 * kMTile * k; q += blockDim.x) {
        const int rr = q / k, a = q - rr * k;
        int pe = -1, ps = -1;
        if (rr < nrows) {
          const int tok = perm[row0 + rr];
          if (tok >= 0 && tok < T) {
            ps = prev.slot_of[static_cast<long long>(tok) * k + a];
            pe = bucket_of(poff, E, ps);
          }
        }
        row_e[q] = pe;
        row_s[q] = ps;
      }
    }
    __syncthreads();
    if (have && warp < kLookupChunks) {
      // warp ch: is chunk ch's run of columns one run of a previous bucket?  The candidates
      // are the first column's previous buckets; each lane looks the candidate up among its
      // own column's k entries (a token's buckets are stored in its routing order).
      const int ch = warp, c = ch * 32 + lane;
      const bool vc = lj0 + c < n_e;
      int fe = -1, fs = 0;
      for (int b = 0; b < k && fe < 0; ++b) {
        const int e0 = __shfl_sync(0xffffffffu, vc ? col_e[c * k + b] : -1, 0);
        const int s0 = __shfl_sync(0xffffffffu, vc ? col_s[c * k + b] : 0, 0);
        if (e0 < 0) continue;
        int my = -1;
        for (int bb = 0; bb < k; ++bb)
          if (vc && col_e[c * k + bb] == e0) my = col_s[c * k + bb];
        if (__all_sync(0xffffffffu, !vc || my == s0 + lane)) {
          fe = e0;
          fs = s0;
        }
      }
      if (lane == 0) {
        s_ch_e[ch] = fe;
        s_ch_s0[ch] = fs;
      }
    }
    __syncthreads();
    bool unknown = false;
    for (int rr = warp; rr < nrows; rr += kLookupThreads / 32) {
      const int li = li0 + rr;
      if (lj0 >= li) continue;  // the row has no pair in this column tile
      const long long wrow = bits_base[e] + static_cast<long long>(li) * W;
      // Word path: lane ch < 8 takes chunk ch when its columns are one run of the previous
      // bucket fe and the row's token was in fe too; its 32 classes are then the 32-bit
      // window of the previous row pi's planes that starts at the run's first slot.
      bool fast = false;
      if (have && lane < kLookupChunks) {
        const int ch = lane;
        const int ljb = lj0 + ch * 32;
        const int fe = s_ch_e[ch];
        if (ljb < li && fe >= 0) {
          int pi = -1;
          for (int a = 0; a < k; ++a)
            if (row_e[rr * k + a] == fe) pi = row_s[rr * k + a];
          const int o = poff[fe];
          const int ne = poff[fe + 1] - o;
          const int nvalid = min(32, li - ljb);
          const int pj0 = s_ch_s0[ch] - o;
          pi -= o;
          if (pi >= 0 && pj0 >= 0 && pj0 + nvalid <= pi && pi < ne) {
            const int Wp = (ne + 31) >> 5;
            const long long base = prev.bits_base[fe] + static_cast<long long>(pi) * Wp;
            const int w0 = pj0 >> 5, sh = pj0 & 31;
            const uint2 lo = prev.planes[base + w0];
            const uint2 hi = (pj0 + nvalid > 32 * (w0 + 1)) ? prev.planes[base + w0 + 1]
                                                              : make_uint2(0u, 0u);
            const unsigned vmask = nvalid == 32 ? 0xffffffffu : (1u << nvalid) - 1u;
            const unsigned kw = __funnelshift_r(lo.x, hi.x, sh) & vmask;
            const unsigned sw = __funnelshift_r(lo.y, hi.y, sh) & kw;
            const long long w = wrow + (ljb >> 5);
            planes_out[w] = make_uint2(kw, sw);
            bits[w] = sw;
            if (sw) atomicMin(&first[row0 + rr], ljb + __ffs(sw) - 1);
            if (kw != vmask) unknown = true;
            fast = true;
          }
        }
      }
      const unsigned fast_chunks = __ballot_sync(0xffffffffu, fast);
      // Lane path for the other chunks: each lane searches its pair's buckets for a common one.
      for (int ch = 0; ch < kLookupChunks; ++ch) {
        const int ljb = lj0 + ch * 32;
        if (ljb >= li) break;
        if ((fast_chunks >> ch) & 1u) continue;
        const int lj = ljb + lane;
        const bool in = lj < li;
        long long widx = -1;
        unsigned bitm = 0u;
        if (have && in) {
          const int c = ch * 32 + lane;
          for (int a = 0; a < k && widx < 0; ++a) {
            const int ea = row_e[rr * k + a];
            if (ea < 0) continue;
            for (int b = 0; b < k; ++b) {
              if (col_e[c * k + b] != ea) continue;
              const int o = poff[ea];
              const int ne = poff[ea + 1] - o;
              const int pi = row_s[rr * k + a] - o, pj = col_s[c * k + b] - o;
              if (pj >= 0 && pj < pi && pi < ne) {
                widx = prev.bits_base[ea] + static_cast<long long>(pi) * ((ne + 31) >> 5) +
                       (pj >> 5);
                bitm = 1u << (pj & 31);
              }
              break;
            }
          }
        }
        const uint2 pv = widx >= 0 ? prev.planes[widx] : make_uint2(0u, 0u);
        const bool kn = in && (pv.x & bitm) != 0u;
        const bool sm = kn && (pv.y & bitm) != 0u;
        const unsigned kw = __ballot_sync(0xffffffffu, kn);
        const unsigned sw = __ballot_sync(0xffffffffu, sm);
        const unsigned iw = __ballot_sync(0xffffffffu, in);
        if (kw != iw) unknown = true;
        if (lane == 0) {
          const long long w = wrow + (ljb >> 5);
          planes_out[w] = make_uint2(kw, sw);
          bits[w] = sw;
          if (sw) atomicMin(&first[row0 + rr], ljb + __ffs(sw) - 1);
        }
      }
    }
    if (unknown && lane == 0) s_unknown = 1;
    __syncthreads();
    if (threadIdx.x == 0 && s_unknown) cos_list[atomicAdd(n_cos, 1)] = tl;
  }
}

// Record header: magic, T, k, E, P.
__global__ void hist_header_kernel(int32_t* header, int T, int k, int E) {
  if (threadIdx.x == 0) {
    header[0] = kHistMagic;
    header[1] = T;
    header[2] = k;
    header[3] = E;
    header[4] = T * k;
  }
}

struct CondenseScratch {
  float* norm;
  unsigned long long* hash;
  int4* mt_info;
  int32_t* group_mt_begin;
  int2* tile_list;
  int32_t* n_list;
  long long* bits_base;
  unsigned* bits;
  int2* cos_list;   // history: tiles with an unclassified pair
  int32_t* n_cos;
  int32_t* overflow;  // a bucket longer than the scratch allows
  int32_t* done;      // greedy-scan CTAs finished (the word after overflow)
  int32_t* first;       // [P] earliest similar row before each row (local), -1 none
  int32_t* unresolved;  // [E] rows the walk has to decide
  int32_t* nrep_fast;   // [E] representatives found without the walk
};

inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Bucket rows the scratch is sized for: a bucket holds each token at most once.
inline int bucket_rows_max(int T, int k) { return T < T * k ? T : T * k; }

size_t carve(void* base, int T, int k, int E, CondenseScratch* s) {
  const int P = T * k;
  const int R = bucket_rows_max(T, k);
  const int n_mt = max_mtiles(P, E);
  const long long max_tiles = static_cast<long long>(n_mt) * ((R + kTcTileN - 1) / kTcTileN);
  const long long max_words = static_cast<long long>(P) * ((R + 31) / 32);
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align256(o + bytes);
    return at;
  };
  const size_t o_norm = take(sizeof(float) * P);
  const size_t o_hash = take(sizeof(unsigned long long) * P);
  const size_t o_mt = take(sizeof(int4) * n_mt);
  const size_t o_gmb = take(sizeof(int32_t) * (E + 1));
  const size_t o_tl = take(sizeof(int2) * max_tiles);
  const size_t o_nl = take(sizeof(int32_t));
  const size_t o_bb = take(sizeof(long long) * E);
  const size_t o_bits = take(sizeof(unsigned) * max_words);
  const size_t o_cl = take(sizeof(int2) * max_tiles);
  const size_t o_nc = take(sizeof(int32_t));
  const size_t o_of = take(sizeof(int32_t) * 2);
  const size_t o_fi = take(sizeof(int32_t) * P);
  const size_t o_un = take(sizeof(int32_t) * E);
  const size_t o_nf = take(sizeof(int32_t) * E);
  if (s && base) {
    char* b = static_cast<char*>(base);
    s->norm = reinterpret_cast<float*>(b + o_norm);
    s->hash = reinterpret_cast<unsigned long long*>(b + o_hash);
    s->mt_info = reinterpret_cast<int4*>(b + o_mt);
    s->group_mt_begin = reinterpret_cast<int32_t*>(b + o_gmb);
    s->tile_list = reinterpret_cast<int2*>(b + o_tl);
    s->n_list = reinterpret_cast<int32_t*>(b + o_nl);
    s->bits_base = reinterpret_cast<long long*>(b + o_bb);
    s->bits = reinterpret_cast<unsigned*>(b + o_bits);
    s->cos_list = reinterpret_cast<int2*>(b + o_cl);
    s->n_cos = reinterpret_cast<int32_t*>(b + o_nc);
    s->overflow = reinterpret_cast<int32_t*>(b + o_of);
    s->done = s->overflow + 1;
    s->first = reinterpret_cast<int32_t*>(b + o_fi);
    s->unresolved = reinterpret_cast<int32_t*>(b + o_un);
    s->nrep_fast = reinterpret_cast<int32_t*>(b + o_nf);
  }
  return o;
}

size_t hist_layout(int T, int k, int E, size_t* at /* 5 offsets or NULL */) {
  const long long P = static_cast<long long>(T) * k;
  const size_t words = static_cast<size_t>(P) * static_cast<size_t>((bucket_rows_max(T, k) + 31) / 32);
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t a = o;
    o = align256(o + bytes);
    return a;
  };
  const size_t a0 = take(sizeof(int32_t) * 5);
  const size_t a1 = take(sizeof(int32_t) * (E + 1));
  const size_t a2 = take(sizeof(int32_t) * static_cast<size_t>(P));
  const size_t a3 = take(sizeof(long long) * E);
  const size_t a4 = take(sizeof(uint2) * words);
  if (at) {
    at[0] = a0; at[1] = a1; at[2] = a2; at[3] = a3; at[4] = a4;
  }
  return o;
}

}  // namespace

size_t condense_scratch_bytes(int T, int k, int E) { return carve(nullptr, T, k, E, nullptr); }

size_t hist_record_bytes(int T, int k, int E) { return hist_layout(T, k, E, nullptr); }

HistView hist_view(const void* base, int T, int k, int E) {
  size_t at[5];
  hist_layout(T, k, E, at);
  char* b = static_cast<char*>(const_cast<void*>(base));
  HistView v;
  v.header = reinterpret_cast<int32_t*>(b + at[0]);
  v.offsets = reinterpret_cast<int32_t*>(b + at[1]);
  v.slot_of = reinterpret_cast<int32_t*>(b + at[2]);
  v.bits_base = reinterpret_cast<long long*>(b + at[3]);
  v.planes = reinterpret_cast<uint2*>(b + at[4]);
  return v;
}

namespace {
cudaError_t condense_pipeline(const __nv_bfloat16* x_perm, const int32_t* offsets, int T, int k,
                              int d, int E, float tau, const HistArgs* h, int num_sms,
                              int32_t* rep_of, int32_t* n_rep, int32_t* n_condensed,
                              void* scratch, unsigned* status, cudaStream_t stream,
                              bool stats_ready);
}  // namespace

cudaError_t launch_condense(const __nv_bfloat16* x_perm, const int32_t* offsets, int T, int k,
                            int d, int E, float tau, int num_sms, int32_t* rep_of, int32_t* n_rep,
                            int32_t* n_condensed, void* scratch, unsigned* status,
                            cudaStream_t stream, bool stats_ready) {
  return condense_pipeline(x_perm, offsets, T, k, d, E, tau, nullptr, num_sms, rep_of, n_rep,
                           n_condensed, scratch, status, stream, stats_ready);
}

cudaError_t launch_condense_hist(const __nv_bfloat16* x_perm, const int32_t* offsets, int d,
                                 int E, float tau, const HistArgs& h, int num_sms,
                                 int32_t* rep_of, int32_t* n_rep, int32_t* n_condensed,
                                 void* scratch, unsigned* status, cudaStream_t stream) {
  return condense_pipeline(x_perm, offsets, h.T, h.k, d, E, tau, &h, num_sms, rep_of, n_rep,
                           n_condensed, scratch, status, stream, false);
}

RowStatsOut condense_stats_ptrs(void* scratch, int T, int k, int E) {
  CondenseScratch s;
  carve(scratch, T, k, E, &s);
  return RowStatsOut{s.norm, s.hash, s.first};
}

namespace {
cudaError_t condense_pipeline(const __nv_bfloat16* x_perm, const int32_t* offsets, int T, int k,
                              int d, int E, float tau, const HistArgs* h, int num_sms,
                              int32_t* rep_of, int32_t* n_rep, int32_t* n_condensed,
                              void* scratch, unsigned* status, cudaStream_t stream,
                              bool stats_ready) {
  const int P = T * k;
  HistView out = {};
  if (h) {
    // the record's header, offsets and slots; its bits_base is written by the tile list
    out = hist_view(h->hist_out, h->T, h->k, E);
    hist_header_kernel<<<1, 32, 0, stream>>>(out.header, h->T, h->k, E);
    cudaError_t e = cudaMemcpyAsync(out.offsets, offsets, sizeof(int32_t) * (E + 1),
                                    cudaMemcpyDeviceToDevice, stream);
    if (e == cudaSuccess && P > 0)
      e = cudaMemcpyAsync(out.slot_of, h->slot_of, sizeof(int32_t) * P, cudaMemcpyDeviceToDevice,
                          stream);
    if (e == cudaSuccess && h->n_cos_tiles)
      e = cudaMemsetAsync(h->n_cos_tiles, 0, sizeof(int32_t), stream);
    if (e != cudaSuccess) return e;
  }
  if (!(tau <= 1.0f) || P == 0) {
    identity_reps_kernel<<<max(1, min(ceil_div(P, 256), 1024)), 256, 0, stream>>>(
        offsets, E, P, rep_of, n_rep, n_condensed);
    if (h) {
      // no pair was compared: every bucket's planes are empty
      cudaError_t e = cudaMemsetAsync(out.bits_base, 0, sizeof(long long) * E, stream);
      if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
  }
  CondenseScratch s;
  carve(scratch, T, k, E, &s);
  cudaError_t err = cudaSuccess;
  if (!stats_ready) {
    err = launch_pdl(row_stats_kernel, dim3(min(ceil_div(P, 8), 4096)), dim3(256), 0, stream,
                     x_perm, offsets, E, d, s.norm, s.hash, s.first);
    if (err != cudaSuccess) return err;
  }
  err = launch_build_mtiles(nullptr, offsets, 0, E, nullptr, s.mt_info, s.group_mt_begin, stream);
  if (err != cudaSuccess) return err;
  long long* bits_base = h ? out.bits_base : s.bits_base;
  err = launch_pdl(sim_tiles_kernel, dim3(1), dim3(256), 0, stream,
                   static_cast<const int4*>(s.mt_info), static_cast<const int32_t*>(s.group_mt_begin),
                   offsets, E, bucket_rows_max(T, k), s.tile_list, s.n_list, bits_base, s.overflow,
                   h ? out.header : nullptr, s.unresolved, s.nrep_fast, s.done, status);
  if (err != cudaSuccess) return err;
  const int2* gemm_list = s.tile_list;
  const int32_t* gemm_n = s.n_list;
  int hist_mode = 0;
  if (h && h->hist_in) {
    // the previous call's classes: tiles whose pairs all have one skip the GEMM
    cudaError_t e = cudaMemsetAsync(s.n_cos, 0, sizeof(int32_t), stream);
    if (e != cudaSuccess) return e;
    const HistView prev = hist_view(h->hist_in, h->T, h->k, E);
    const size_t smem = sizeof(int) * ((E + 1) + 2 * (kTcTileN + 2 * kMTile) * h->k);
    static OncePerDevice<64> once_l;
    int dev = 0;
    cudaGetDevice(&dev);
    e = once_l.run(dev, [&]() {
      // the largest table: E = 256, k = 32
      return cudaFuncSetAttribute(hist_lookup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(sizeof(int) * (257 + 2 * (kTcTileN + 2 * kMTile) * 32)));
    });
    if (e != cudaSuccess) return e;
    const int max_tiles = max_mtiles(P, E) * ((bucket_rows_max(T, k) + kTcTileN - 1) / kTcTileN);
    hist_lookup_kernel<<<max(1, min(max_tiles, 8 * num_sms)), kLookupThreads, smem, stream>>>(
        s.tile_list, s.n_list, s.mt_info, offsets, h->perm, h->T, h->k, E, bits_base, prev,
        out.planes, s.bits, s.first, s.cos_list, s.n_cos);
    gemm_list = s.cos_list;
    gemm_n = s.n_cos;
    hist_mode = 2;
  } else if (h) {
    hist_mode = 1;
  }
  if (h && h->n_cos_tiles) {
    cudaError_t e = cudaMemcpyAsync(h->n_cos_tiles, gemm_n, sizeof(int32_t),
                                    cudaMemcpyDeviceToDevice, stream);
    if (e != cudaSuccess) return e;
  }
  TcGemmArgs a = {};
  a.mt_info = s.mt_info;
  a.group_mt_begin = s.group_mt_begin;
  a.n_groups = E;
  a.tile_list = gemm_list;
  a.n_list = gemm_n;
  a.hist_mode = hist_mode;
  a.hplanes = out.planes;
  a.s1 = h ? h->s1 : 2.0f;
  a.s2 = h ? h->s2 : -2.0f;
  a.n_kblocks = d / kTcTileK;
  a.kb_per_slice = a.n_kblocks;
  a.nt_per_slice = 1;
  a.norm = s.norm;
  a.row_hash = s.hash;
  a.rows = x_perm;
  a.d = d;
  a.bucket_off = offsets;
  a.bits_base = bits_base;
  a.bits = s.bits;
  a.tau = tau;
  a.first = s.first;
  a.status = status;
  err = tc_gemm(kTcSimBits, x_perm, P, d, x_perm, 1, P, d, a, num_sms, stream);
  if (err != cudaSuccess) return err;
  const size_t smem = sizeof(unsigned) * (kMaxWords + 2 * kScanBufWords);
  // the shared-memory limit is a per-device attribute of the function
  static OncePerDevice<64> once;
  int dev = 0;
  cudaGetDevice(&dev);
  err = once.run(dev, [&]() {
    return cudaFuncSetAttribute(greedy_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(smem));
  });
  if (err != cudaSuccess) return err;
  err = launch_pdl(resolve_kernel, dim3(max(1, min(ceil_div(P, 256), 4 * num_sms))), dim3(256), 0,
                   stream, static_cast<const int32_t*>(s.first), offsets, E,
                   static_cast<const int32_t*>(s.overflow), rep_of, s.unresolved, s.nrep_fast);
  if (err != cudaSuccess) return err;
  err = launch_pdl(greedy_scan_kernel, dim3(E), dim3(kScanThreads), smem, stream,
                   static_cast<const unsigned*>(s.bits), static_cast<const long long*>(bits_base),
                   offsets, static_cast<const int32_t*>(s.overflow),
                   static_cast<const int32_t*>(s.unresolved),
                   static_cast<const int32_t*>(s.nrep_fast), rep_of, n_rep, s.done, n_condensed,
                   status);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_compact_reps(const int32_t* rep_of, const int32_t* offsets, int E,
                                int32_t* rep_local, int32_t* rep_counts, cudaStream_t stream) {
  const cudaError_t e = launch_pdl(compact_reps_kernel, dim3(E), dim3(1024), 0, stream, rep_of,
                                   offsets, E, rep_local, rep_counts);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_gather_reps(int act_dtype, const void* src, const int32_t* rep_local,
                               const int32_t* offsets, const int32_t* rep_off, int E, int max_rows,
                               int d, void* dst, int32_t* rep_rows, cudaStream_t stream) {
  if (max_rows <= 0) return cudaSuccess;
  const int blocks = min(ceil_div(max_rows, 8), 4096);
  const cudaError_t e =
      act_dtype == MOE_F32
          ? launch_pdl(gather_reps_kernel<float>, dim3(blocks), dim3(256), 0, stream,
                       static_cast<const float*>(src), rep_local, offsets, rep_off, E, d,
                       static_cast<float*>(dst), rep_rows)
          : launch_pdl(gather_reps_kernel<__nv_bfloat16>, dim3(blocks), dim3(256), 0, stream,
                       static_cast<const __nv_bfloat16*>(src), rep_local, offsets, rep_off, E, d,
                       static_cast<__nv_bfloat16*>(dst), rep_rows);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace moe
