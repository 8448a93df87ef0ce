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
// Determinism: slot ranks come from per-chunk counts, an exclusive scan over
// (expert, chunk), and an in-chunk ordered rank (warp match + popc), so the
// permutation is the same on every run; the combine sums in a fixed order.
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

// One CTA: expert totals, offsets, and the first slot of every (expert, chunk).
__global__ void __launch_bounds__(256)
    dispatch_scan_kernel(const int32_t* __restrict__ chunk_counts, int E, int n_chunks,
                         int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                         int32_t* __restrict__ chunk_base) {
  __shared__ int s_cnt[256];
  __shared__ int s_off[257];
  const int e = threadIdx.x;
  if (e < E) {
    int tot = 0;
    for (int c = 0; c < n_chunks; ++c) tot += chunk_counts[static_cast<long long>(e) * n_chunks + c];
    s_cnt[e] = tot;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0;
    for (int i = 0; i < E; ++i) {
      s_off[i] = run;
      run += s_cnt[i];
    }
    s_off[E] = run;
  }
  __syncthreads();
  if (e < E) {
    counts[e] = s_cnt[e];
    offsets[e] = s_off[e];
    int run = s_off[e];
    for (int c = 0; c < n_chunks; ++c) {
      chunk_base[static_cast<long long>(e) * n_chunks + c] = run;
      run += chunk_counts[static_cast<long long>(e) * n_chunks + c];
    }
  }
  if (threadIdx.x == 0) offsets[E] = s_off[E];
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
    int slot = 0;
    if (e >= 0) {
      slot = base[e] + __popc(peers & lt);
      perm[slot] = static_cast<int32_t>(p / k);
      slot_of[p] = slot;
    }
    __syncwarp();
    if (e >= 0 && lane == 31 - __clz(peers)) base[e] += __popc(peers);
    __syncwarp();
  }
}

// dst[r] = src[rows[r]] for r < *n_rows_dev; one warp per row, 16-byte vectors.
template <typename T>
__global__ void __launch_bounds__(256)
    gather_rows_kernel(const T* __restrict__ src, const int32_t* __restrict__ rows,
                       const int* __restrict__ n_rows_dev, int src_rows, int d,
                       T* __restrict__ dst, unsigned* status) {
  constexpr int V = Act<T>::kVec;
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
template <typename T>
__global__ void __launch_bounds__(128)
    combine_kernel(const T* __restrict__ y, const T* __restrict__ shared_out,
                   const int32_t* __restrict__ slot_of, const int32_t* __restrict__ rep_of,
                   const float* __restrict__ gate, const T* __restrict__ x,
                   const T* residual, int residual_mode, T* out, int d, int k, int P,
                   unsigned* status) {
  constexpr int V = Act<T>::kVec;
  __shared__ long long s_row[32];
  __shared__ float s_g[32];
  const int t = blockIdx.x;
  if (threadIdx.x < k) {
    int s = slot_of[static_cast<long long>(t) * k + threadIdx.x];
    if (s >= 0 && s < P && rep_of) s = rep_of[s];
    if (s < 0 || s >= P) {
      record_status(status, MOE_ERR_DEVICE_INDEX);
      s = -1;
    }
    s_row[threadIdx.x] = s;
    s_g[threadIdx.x] = gate[static_cast<long long>(t) * k + threadIdx.x];
  }
  __syncthreads();
  const long long rowoff = static_cast<long long>(t) * d;
  for (int v = threadIdx.x; v < d / V; v += blockDim.x) {
    float acc[V], tmp[V];
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = 0.f;
    if (residual_mode == MOE_RES_INPUT || residual_mode == MOE_RES_INPUT_PLUS_EXTERNAL) {
      load_vec_f32<T>(x + rowoff + v * V, tmp);
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] += tmp[i];
    }
    if (residual_mode == MOE_RES_EXTERNAL || residual_mode == MOE_RES_INPUT_PLUS_EXTERNAL) {
      load_vec_f32<T>(residual + rowoff + v * V, tmp);
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] += tmp[i];
    }
    if (shared_out) {
      load_vec_f32<T>(shared_out + rowoff + v * V, tmp);
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] += tmp[i];
    }
    for (int j = 0; j < k; ++j) {
      const long long s = s_row[j];
      if (s < 0) continue;
      const float g = s_g[j];
      load_vec_f32<T>(y + s * d + v * V, tmp);
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] = fmaf(g, tmp[i], acc[i]);
    }
    store_vec_f32<T>(out + rowoff + v * V, acc);
  }
}

__global__ void __launch_bounds__(256)
    build_mtiles_kernel(const int32_t* __restrict__ counts, const int32_t* __restrict__ offsets_in,
                        int fixed_rows, int n_groups,
                        int32_t* __restrict__ offsets_out, int4* __restrict__ mt_info,
                        int32_t* __restrict__ group_mt_begin) {
  __shared__ int s_rows[256];
  __shared__ int s_off[257];
  __shared__ int s_mt[257];
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
  dispatch_scan_kernel<<<1, 256, 0, stream>>>(chunk_counts, E, n_chunks, counts, offsets,
                                              chunk_base);
  if (T == 0) return cudaGetLastError();
  dispatch_scatter_kernel<<<n_chunks, kScatterThreads, 0, stream>>>(topk_idx, T, E, k, n_chunks, chunk_base,
                                                       perm, slot_of);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_gather_rows(act_dtype, x, T, perm, offsets + E, T * k, d, x_perm, status, stream);
}

cudaError_t launch_gather_rows(int act_dtype, const void* src, int src_rows, const int32_t* rows,
                               const int* n_rows_dev, int max_rows, int d, void* dst,
                               unsigned* status, cudaStream_t stream) {
  if (max_rows <= 0) return cudaSuccess;
  const int blocks = min(ceil_div(max_rows, 8), 4096);
  if (act_dtype == MOE_F32)
    gather_rows_kernel<float><<<blocks, 256, 0, stream>>>(
        static_cast<const float*>(src), rows, n_rows_dev, src_rows, d, static_cast<float*>(dst),
        status);
  else
    gather_rows_kernel<__nv_bfloat16><<<blocks, 256, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(src), rows, n_rows_dev, src_rows, d,
        static_cast<__nv_bfloat16*>(dst), status);
  return cudaGetLastError();
}

cudaError_t launch_combine(int act_dtype, const void* y_perm, const void* shared_out,
                           const int32_t* slot_of, const int32_t* rep_of, const float* topk_gate,
                           const void* x, const void* residual, int residual_mode, void* out, int T,
                           int d, int k, int P, unsigned* status, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  if (act_dtype == MOE_F32)
    combine_kernel<float><<<T, 128, 0, stream>>>(
        static_cast<const float*>(y_perm), static_cast<const float*>(shared_out), slot_of, rep_of,
        topk_gate, static_cast<const float*>(x), static_cast<const float*>(residual),
        residual_mode, static_cast<float*>(out), d, k, P, status);
  else
    combine_kernel<__nv_bfloat16><<<T, 128, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(y_perm), static_cast<const __nv_bfloat16*>(shared_out),
        slot_of, rep_of, topk_gate, static_cast<const __nv_bfloat16*>(x),
        static_cast<const __nv_bfloat16*>(residual), residual_mode,
        static_cast<__nv_bfloat16*>(out), d, k, P, status);
  return cudaGetLastError();
}

cudaError_t launch_build_mtiles(const int32_t* counts, const int32_t* offsets_in, int fixed_rows,
                                int n_groups, int32_t* offsets_out, int4* mt_info,
                                int32_t* group_mt_begin, cudaStream_t stream) {
  build_mtiles_kernel<<<1, 256, 0, stream>>>(counts, offsets_in, fixed_rows, n_groups, offsets_out,
                                             mt_info, group_mt_begin);
  return cudaGetLastError();
}

}  // namespace moe
