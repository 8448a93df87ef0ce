// Kernels around the backward GEMMs of the routed-expert layer (gemm_bwd.cu):
// the padded slot space, the recomputed SwiGLU activations, the combine's and
// the router's backward, the router's small fp32 products and the assembly of
// the input gradient.  Everything is deterministic: no atomics, every sum in
// a fixed order.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kPad = 64;  // rows of a group in the padded slot space start at a multiple of this

__global__ void pad_counts_kernel(const int32_t* __restrict__ counts, int E,
                                  int32_t* __restrict__ pcounts) {
  pdl_trigger();
  pdl_wait();
  for (int e = threadIdx.x; e < E; e += blockDim.x) pcounts[e] = (counts[e] + kPad - 1) & ~(kPad - 1);
}

// One warp per padded row q < poffsets[E]: x_pad[q] = x_perm[src] for a real row of group e,
// src = offsets[e] + q - poffsets[e] (or its representative rep_of[src] when condensing: a
// condensed slot's expert input is its representative's row), zeros for a pad row (whose
// dy_pad row is zeroed as well).
template <typename T>
__global__ void __launch_bounds__(256)
    pad_rows_kernel(const T* __restrict__ x_perm, const int32_t* __restrict__ offsets,
                    const int32_t* __restrict__ poffsets, const int32_t* __restrict__ rep_of,
                    int E, int max_rows, int d, T* __restrict__ x_pad, T* __restrict__ dy_pad) {
  pdl_trigger();
  pdl_wait();
  const int total = poffsets[E];
  const int nv = d * static_cast<int>(sizeof(T)) / 16;
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int q = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; q < total && q < max_rows; q += warps) {
    int lo = 0, hi = E;  // largest e with poffsets[e] <= q
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (poffsets[mid] <= q) lo = mid; else hi = mid;
    }
    const int i = q - poffsets[lo];
    uint4* dst = reinterpret_cast<uint4*>(x_pad + static_cast<long long>(q) * d);
    if (i < offsets[lo + 1] - offsets[lo]) {
      int slot = offsets[lo] + i;
      if (rep_of) slot = rep_of[slot];
      const uint4* src = reinterpret_cast<const uint4*>(x_perm + static_cast<long long>(slot) * d);
      for (int v = lane; v < nv; v += 32) dst[v] = src[v];
    } else {
      uint4* dz = reinterpret_cast<uint4*>(dy_pad + static_cast<long long>(q) * d);
      for (int v = lane; v < nv; v += 32) dst[v] = dz[v] = make_uint4(0, 0, 0, 0);
    }
  }
}

// dst[t] = src[t] for t < T, zeros for T <= t < T_pad (one warp per row).
template <typename T>
__global__ void __launch_bounds__(256)
    pad_tokens_kernel(const T* __restrict__ src, int T_tok, int T_pad, int d, T* __restrict__ dst) {
  pdl_trigger();
  pdl_wait();
  const int nv = d * static_cast<int>(sizeof(T)) / 16;
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T_pad; t += warps) {
    uint4* o = reinterpret_cast<uint4*>(dst + static_cast<long long>(t) * d);
    if (t < T_tok) {
      const uint4* s = reinterpret_cast<const uint4*>(src + static_cast<long long>(t) * d);
      for (int v = lane; v < nv; v += 32) o[v] = s[v];
    } else {
      for (int v = lane; v < nv; v += 32) o[v] = make_uint4(0, 0, 0, 0);
    }
  }
}

// h[row][s][i] = SiLU(a) * u with [a | u] = au[row][s][0..2Hs) (bf16 in, bf16 out).
// Rows on blockIdx.y (grid-strided), 8 hidden units (16 bytes) per thread.
__global__ void __launch_bounds__(256)
    swiglu_from_au_kernel(const __nv_bfloat16* __restrict__ au, const int* __restrict__ n_rows_dev,
                          int rows_max, int S, int Hs, __nv_bfloat16* __restrict__ h) {
  pdl_trigger();
  pdl_wait();
  const int rows = n_rows_dev ? min(*n_rows_dev, rows_max) : rows_max;
  const int vec_per_row = S * Hs / 8;
  for (int row = blockIdx.y; row < rows; row += gridDim.y) {
    for (int v = blockIdx.x * blockDim.x + threadIdx.x; v < vec_per_row; v += gridDim.x * blockDim.x) {
      const int s = (v * 8) / Hs;
      const int col = v * 8 - s * Hs;
      const __nv_bfloat16* base = au + static_cast<long long>(row) * 2 * S * Hs + s * 2 * Hs + col;
      const uint4 av = *reinterpret_cast<const uint4*>(base);
      const uint4 uv = *reinterpret_cast<const uint4*>(base + Hs);
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&av);
      const __nv_bfloat162* u2 = reinterpret_cast<const __nv_bfloat162*>(&uv);
      uint4 out;
      __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(&out);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 a = __bfloat1622float2(a2[i]);
        const float2 u = __bfloat1622float2(u2[i]);
        o2[i] = __floats2bfloat162_rn(a.x / (1.0f + __expf(-a.x)) * u.x,
                                      a.y / (1.0f + __expf(-a.y)) * u.y);
      }
      *reinterpret_cast<uint4*>(h + static_cast<long long>(row) * S * Hs + v * 8) = out;
    }
  }
}

// Combine backward, one CTA per token (one 16-byte vector per thread):
//   dg[t, j] = <d_out[t], y[slot]>          (fp32, summed in a fixed order)
//   dy_pad[slot] = gate[t, j] * d_out[t]    (bf16)
// slot = the pair's row in the padded slot space.
template <typename T>
__global__ void __launch_bounds__(256)
    combine_bwd_kernel(const T* __restrict__ d_out, const T* __restrict__ y_pad,
                       const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ slot_of,
                       const int32_t* __restrict__ offsets, const int32_t* __restrict__ poffsets,
                       const float* __restrict__ gate, int d, int k, T* __restrict__ dy_pad,
                       float* __restrict__ dg) {
  constexpr int V = Act<T>::kVec;
  __shared__ long long s_row[32];
  __shared__ float s_part[32][33];
  const int t = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  pdl_trigger();
  pdl_wait();
  if (threadIdx.x < k) {
    const long long p = static_cast<long long>(t) * k + threadIdx.x;
    const int e = topk_idx[p];
    const int s = slot_of[p];
    s_row[threadIdx.x] = (s >= 0) ? static_cast<long long>(s - offsets[e] + poffsets[e]) : -1;
  }
  __syncthreads();
  float part[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) part[j] = 0.f;
  const long long rowoff = static_cast<long long>(t) * d;
  for (int v = threadIdx.x; v < d / V; v += blockDim.x) {
    float o[V], yv[V];
    load_vec_f32<T>(d_out + rowoff + v * V, o);
    for (int j = 0; j < k; ++j) {
      const long long s = s_row[j];
      if (s < 0) continue;
      load_vec_f32<T>(y_pad + s * d + v * V, yv);
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < V; ++i) acc = fmaf(o[i], yv[i], acc);
      part[j] += acc;
      const float g = gate[static_cast<long long>(t) * k + j];
      float w[V];
#pragma unroll
      for (int i = 0; i < V; ++i) w[i] = g * o[i];
      store_vec_f32<T>(dy_pad + s * d + v * V, w);
    }
  }
  for (int j = 0; j < k; ++j) {
    float x = part[j];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    if (lane == 0) s_part[j][warp] = x;
  }
  __syncthreads();
  if (threadIdx.x < k) {
    float sum = 0.f;
    for (int w = 0; w < nwarps; ++w) sum += s_part[threadIdx.x][w];
    dg[static_cast<long long>(t) * k + threadIdx.x] = s_row[threadIdx.x] >= 0 ? sum : 0.f;
  }
}

// Router backward, one warp per token: dlogits from the gate gradients (the
// top-k selection passes no gradient).
__global__ void __launch_bounds__(256)
    router_bwd_kernel(const float* __restrict__ logits, const int32_t* __restrict__ topk_idx,
                      const float* __restrict__ gate, const float* __restrict__ dg, int T, int E,
                      int k, int gating, float* __restrict__ dl) {
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  pdl_trigger();
  pdl_wait();
  if (t >= T) return;
  const float* l = logits + static_cast<long long>(t) * E;
  float* o = dl + static_cast<long long>(t) * E;
  const int32_t* ix = topk_idx + static_cast<long long>(t) * k;
  const float* g = gate + static_cast<long long>(t) * k;
  const float* dgt = dg + static_cast<long long>(t) * k;
  if (gating == MOE_GATE_SOFTMAX_TOPK) {
    // p = softmax(l) over all E; dl = p * (dp - <dp, p>), dp[e_j] = dg_j
    float m = -INFINITY;
    for (int e = lane; e < E; e += 32) m = fmaxf(m, l[e]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    float z = 0.f;
    for (int e = lane; e < E; e += 32) z += expf(l[e] - m);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
    float dot = 0.f;  // <dp, p> = sum_j dg_j p[e_j] = sum_j dg_j g_j
    for (int j = 0; j < k; ++j) dot += dgt[j] * g[j];
    for (int e = lane; e < E; e += 32) {
      float dp = 0.f;
      for (int j = 0; j < k; ++j)
        if (ix[j] == e) dp = dgt[j];
      const float p = expf(l[e] - m) / z;
      o[e] = p * (dp - dot);
    }
  } else {
    for (int e = lane; e < E; e += 32) o[e] = 0.f;
    __syncwarp();
    if (lane < k) {
      float v;
      if (gating == MOE_GATE_SOFTMAX_TOPK_RENORM) {
        float dot = 0.f;
        for (int j = 0; j < k; ++j) dot += dgt[j] * g[j];
        v = g[lane] * (dgt[lane] - dot);
      } else {
        v = dgt[lane] * g[lane] * (1.0f - g[lane]);
      }
      o[ix[lane]] = v;
    }
  }
}

// C[z][m][n] = sum_{k in split z} A(m, k) B(k, n), fp32 FMA; 64 x 64 tiles, 16-deep
// K steps.  A(m, k) = A[m * sam + k * sak]; B(k, n) = B[k * sbk + n * sbn].
// KFAST: the staging loads walk K fastest (operands contiguous along K), else M/N fastest.
template <typename TA, bool KFAST>
__global__ void __launch_bounds__(256)
    small_gemm_kernel(const TA* __restrict__ A, long long sam, long long sak,
                      const float* __restrict__ B, long long sbk, long long sbn, int M, int N,
                      int K, int k_len, float* __restrict__ C) {
  __shared__ float As[16][65];
  __shared__ float Bs[16][65];
  pdl_trigger();
  pdl_wait();
  const int m0 = blockIdx.x * 64, n0 = blockIdx.y * 64;
  const int k_begin = blockIdx.z * k_len, k_end = min(K, k_begin + k_len);
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4] = {};
  for (int k0 = k_begin; k0 < k_end; k0 += 16) {
    for (int i = threadIdx.x; i < 16 * 64; i += 256) {
      const int kk = KFAST ? (i & 15) : (i >> 6), mm = KFAST ? (i >> 4) : (i & 63);
      const int gk = k0 + kk;
      As[kk][mm] = (gk < k_end && m0 + mm < M)
                       ? Act<TA>::to_f(A[(m0 + mm) * sam + static_cast<long long>(gk) * sak])
                       : 0.f;
      Bs[kk][mm] = (gk < k_end && n0 + mm < N) ? B[static_cast<long long>(gk) * sbk + (n0 + mm) * sbn] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i], b[i] = Bs[kk][tx * 4 + i];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
  float* c = C + static_cast<long long>(blockIdx.z) * M * N;
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int m = m0 + ty * 4 + i, n = n0 + tx * 4 + j;
      if (m < M && n < N) c[static_cast<long long>(m) * N + n] = acc[i][j];
    }
}

// out[i] = sum_z part[z][i] (z in order); also, when col_sums is given, col_sums[n] =
// sum over rows of src [rows][N] in row order (the bias gradient).
__global__ void __launch_bounds__(256)
    reduce_splits_kernel(const float* __restrict__ part, int n_split, long long n, float* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    float s = part[i];
    for (int z = 1; z < n_split; ++z) s += part[static_cast<long long>(z) * n + i];
    out[i] = s;
  }
}

// part[b][n] = sum of src rows [64 b, 64 b + 64) of column n (rows in order).
__global__ void __launch_bounds__(256)
    column_partials_kernel(const float* __restrict__ src, int rows, int N, float* __restrict__ part) {
  pdl_trigger();
  pdl_wait();
  const int r0 = blockIdx.x * 64, r1 = min(rows, r0 + 64);
  for (int n = threadIdx.x; n < N; n += blockDim.x) {
    float s = 0.f;
    for (int r = r0; r < r1; ++r) s += src[static_cast<long long>(r) * N + n];
    part[static_cast<long long>(blockIdx.x) * N + n] = s;
  }
}

// Members of every representative slot (the slots condensed onto it), in ascending slot
// order: mem_list[mem_off[r] .. mem_off[r] + mem_cnt[r]).  One CTA per bucket; thread 0
// counts and fills sequentially; bucket e's lists lie inside [offsets[e], offsets[e+1])
// (a bucket has fewer members than slots), so buckets never share an entry.
__global__ void __launch_bounds__(32)
    members_kernel(const int32_t* __restrict__ rep_of, const int32_t* __restrict__ offsets,
                   int32_t* __restrict__ mem_off, int32_t* __restrict__ mem_cnt,
                   int32_t* __restrict__ mem_list) {
  pdl_trigger();
  pdl_wait();
  if (threadIdx.x != 0) return;
  const int a = offsets[blockIdx.x], b = offsets[blockIdx.x + 1];
  for (int s = a; s < b; ++s) mem_cnt[s] = 0;
  for (int s = a; s < b; ++s)
    if (rep_of[s] != s) ++mem_cnt[rep_of[s]];
  int run = a;
  for (int s = a; s < b; ++s) {
    mem_off[s] = run;
    run += mem_cnt[s];
  }
  for (int s = a; s < b; ++s) {
    const int r = rep_of[s];
    if (r != s) mem_list[mem_off[r]++] = s;  // mem_off[r] runs as the fill cursor ...
  }
  for (int s = a; s < b; ++s) mem_off[s] -= mem_cnt[s];  // ... and is moved back to the start
}

// dx[t] = [d_out[t] if the residual is x] + dx_router[t] + dz_shared[t] + sum_j dz[slot(t, j)],
// fp32 in that order, rounded once.  With condensation the expert-input gradient of a slot
// belongs to the token whose row the slot read: a representative slot of t adds its own dz
// and then its members' dz (ascending slot), a condensed slot of t adds nothing.
// One CTA per token, 4 fp32 per thread.
template <typename T>
__global__ void __launch_bounds__(256)
    dx_assemble_kernel(const T* __restrict__ d_out, int add_dout, const float* __restrict__ dx_router,
                       const float* __restrict__ dz_shared, const float* __restrict__ dz,
                       const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ slot_of,
                       const int32_t* __restrict__ offsets, const int32_t* __restrict__ poffsets,
                       const int32_t* __restrict__ rep_of, const int32_t* __restrict__ mem_off,
                       const int32_t* __restrict__ mem_cnt, const int32_t* __restrict__ mem_list,
                       int d, int k, T* __restrict__ dx) {
  __shared__ long long s_row[32];
  __shared__ int s_mem[32][2];  // member range of each pair's slot (representatives only)
  __shared__ int s_shift[32];   // padded-row shift of the pair's bucket
  const int t = blockIdx.x;
  pdl_trigger();
  pdl_wait();
  if (threadIdx.x < k) {
    const long long p = static_cast<long long>(t) * k + threadIdx.x;
    const int s = slot_of[p];
    const int e = topk_idx[p];
    const int shift = s >= 0 ? poffsets[e] - offsets[e] : 0;
    s_shift[threadIdx.x] = shift;
    s_mem[threadIdx.x][0] = s_mem[threadIdx.x][1] = 0;
    if (s >= 0 && rep_of && rep_of[s] != s) {
      s_row[threadIdx.x] = -1;  // condensed: its gradient went to the representative's token
    } else {
      s_row[threadIdx.x] = s >= 0 ? static_cast<long long>(s + shift) : -1;
      if (s >= 0 && rep_of) {
        s_mem[threadIdx.x][0] = mem_off[s];
        s_mem[threadIdx.x][1] = mem_off[s] + mem_cnt[s];
      }
    }
  }
  __syncthreads();
  const long long rowoff = static_cast<long long>(t) * d;
  for (int c = threadIdx.x * 4; c < d; c += blockDim.x * 4) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if (add_dout) {
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[i] += Act<T>::to_f(d_out[rowoff + c + i]);
    }
    const float4 r = *reinterpret_cast<const float4*>(dx_router + rowoff + c);
    acc[0] += r.x; acc[1] += r.y; acc[2] += r.z; acc[3] += r.w;
    if (dz_shared) {
      const float4 s = *reinterpret_cast<const float4*>(dz_shared + rowoff + c);
      acc[0] += s.x; acc[1] += s.y; acc[2] += s.z; acc[3] += s.w;
    }
    for (int j = 0; j < k; ++j) {
      const long long s = s_row[j];
      if (s < 0) continue;
      const float4 z = *reinterpret_cast<const float4*>(dz + s * d + c);
      acc[0] += z.x; acc[1] += z.y; acc[2] += z.z; acc[3] += z.w;
      for (int m = s_mem[j][0]; m < s_mem[j][1]; ++m) {
        const long long ms = static_cast<long long>(mem_list[m]) + s_shift[j];
        const float4 w = *reinterpret_cast<const float4*>(dz + ms * d + c);
        acc[0] += w.x; acc[1] += w.y; acc[2] += w.z; acc[3] += w.w;
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) dx[rowoff + c + i] = Act<T>::from_f(acc[i]);
  }
}

}  // namespace

cudaError_t launch_pad_counts(const int32_t* counts, int E, int32_t* pcounts, cudaStream_t st) {
  return launch_pdl(pad_counts_kernel, dim3(1), dim3(256), 0, st, counts, E, pcounts);
}

cudaError_t launch_pad_rows(const void* x_perm, const int32_t* offsets, const int32_t* poffsets,
                            const int32_t* rep_of, int E, int max_rows, int d, void* x_pad,
                            void* dy_pad, cudaStream_t st) {
  const int blocks = min(ceil_div(max_rows, 8), 8192);
  return launch_pdl(pad_rows_kernel<__nv_bfloat16>, dim3(blocks), dim3(256), 0, st,
                    static_cast<const __nv_bfloat16*>(x_perm), offsets, poffsets, rep_of, E,
                    max_rows, d, static_cast<__nv_bfloat16*>(x_pad),
                    static_cast<__nv_bfloat16*>(dy_pad));
}

cudaError_t launch_pad_tokens(const void* src, int T, int T_pad, int d, void* dst,
                              cudaStream_t st) {
  const int blocks = min(ceil_div(T_pad, 8), 8192);
  return launch_pdl(pad_tokens_kernel<__nv_bfloat16>, dim3(blocks), dim3(256), 0, st,
                    static_cast<const __nv_bfloat16*>(src), T, T_pad, d,
                    static_cast<__nv_bfloat16*>(dst));
}

cudaError_t launch_swiglu_from_au(const void* au, const int* n_rows_dev, int rows_max, int S,
                                  int Hs, void* h, cudaStream_t st) {
  const int vec_per_row = S * Hs / 8;
  const int gx = ceil_div(vec_per_row, 256);
  const int gy = max(1, min(rows_max, 65535));
  return launch_pdl(swiglu_from_au_kernel, dim3(gx, gy), dim3(256), 0, st,
                    static_cast<const __nv_bfloat16*>(au), n_rows_dev, rows_max, S, Hs,
                    static_cast<__nv_bfloat16*>(h));
}

cudaError_t launch_combine_bwd(const void* d_out, const void* y_pad, const int32_t* topk_idx,
                               const int32_t* slot_of, const int32_t* offsets,
                               const int32_t* poffsets, const float* gate, int T, int d, int k,
                               void* dy_pad, float* dg, cudaStream_t st) {
  const int threads = min(256, max(32, ceil_div(d / 8, 32) * 32));
  return launch_pdl(combine_bwd_kernel<__nv_bfloat16>, dim3(T), dim3(threads), 0, st,
                    static_cast<const __nv_bfloat16*>(d_out),
                    static_cast<const __nv_bfloat16*>(y_pad), topk_idx, slot_of, offsets,
                    poffsets, gate, d, k, static_cast<__nv_bfloat16*>(dy_pad), dg);
}

cudaError_t launch_router_bwd(const float* logits, const int32_t* topk_idx, const float* gate,
                              const float* dg, int T, int E, int k, int gating, float* dl,
                              cudaStream_t st) {
  return launch_pdl(router_bwd_kernel, dim3(ceil_div(T, 8)), dim3(256), 0, st, logits, topk_idx,
                    gate, dg, T, E, k, gating, dl);
}

size_t router_bwd_scratch_bytes(int T, int d, int E) {
  const int splits = max(1, min(64, T / 256));
  const size_t a = static_cast<size_t>(splits) * d * E * sizeof(float);
  const size_t b = static_cast<size_t>(ceil_div(T, 64)) * E * sizeof(float);
  return a > b ? a : b;
}

cudaError_t launch_router_param_grads(const void* x, const float* dl, const float* W_r, int T,
                                      int d, int E, float* dW_r, float* d_bias, float* dx_router,
                                      void* scratch, cudaStream_t st) {
  // dx_router[T][d] = dl[T][E] . W_r^T   (W_r is [d][E])
  cudaError_t err = launch_pdl(small_gemm_kernel<float, true>, dim3(ceil_div(T, 64), ceil_div(d, 64), 1),
                               dim3(256), 0, st, dl, static_cast<long long>(E), 1ll, W_r, 1ll,
                               static_cast<long long>(E), T, d, E, E, dx_router);
  if (err != cudaSuccess) return err;
  // dW_r[d][E] = x^T . dl, split over the T rows, partials summed in order
  const int splits = max(1, min(64, T / 256));
  const int k_len = ceil_div(ceil_div(T, splits), 16) * 16;
  const int n_split = ceil_div(T, k_len);
  float* part = static_cast<float*>(scratch);
  err = launch_pdl(small_gemm_kernel<__nv_bfloat16, false>, dim3(ceil_div(d, 64), ceil_div(E, 64), n_split),
                   dim3(256), 0, st, static_cast<const __nv_bfloat16*>(x), 1ll,
                   static_cast<long long>(d), dl, static_cast<long long>(E), 1ll, d, E, T, k_len,
                   part);
  if (err != cudaSuccess) return err;
  const long long n = static_cast<long long>(d) * E;
  err = launch_pdl(reduce_splits_kernel, dim3(static_cast<int>(min(4096ll, (n + 255) / 256))),
                   dim3(256), 0, st, static_cast<const float*>(part), n_split, n, dW_r);
  if (err != cudaSuccess) return err;
  if (d_bias) {
    // bias gradient: column sums of dl over the T rows, 64-row partials summed in order
    // (the scratch is free again: the stream has finished the dW_r reduction first)
    const int nb = ceil_div(T, 64);
    err = launch_pdl(column_partials_kernel, dim3(nb), dim3(256), 0, st, dl, T, E, part);
    if (err != cudaSuccess) return err;
    err = launch_pdl(reduce_splits_kernel, dim3(ceil_div(E, 256)), dim3(256), 0, st,
                     static_cast<const float*>(part), nb, static_cast<long long>(E), d_bias);
  }
  return err;
}

cudaError_t launch_members(const int32_t* rep_of, const int32_t* offsets, int E, int32_t* mem_off,
                           int32_t* mem_cnt, int32_t* mem_list, cudaStream_t st) {
  return launch_pdl(members_kernel, dim3(E), dim3(32), 0, st, rep_of, offsets, mem_off, mem_cnt,
                    mem_list);
}

cudaError_t launch_dx_assemble(const void* d_out, int add_dout, const float* dx_router,
                               const float* dz_shared, const float* dz, const int32_t* topk_idx,
                               const int32_t* slot_of, const int32_t* offsets,
                               const int32_t* poffsets, const int32_t* rep_of,
                               const int32_t* mem_off, const int32_t* mem_cnt,
                               const int32_t* mem_list, int T, int d, int k, void* dx,
                               cudaStream_t st) {
  const int threads = min(256, max(32, ceil_div(d / 4, 32) * 32));
  return launch_pdl(dx_assemble_kernel<__nv_bfloat16>, dim3(T), dim3(threads), 0, st,
                    static_cast<const __nv_bfloat16*>(d_out), add_dout, dx_router, dz_shared, dz,
                    topk_idx, slot_of, offsets, poffsets, rep_of, mem_off, mem_cnt, mem_list, d,
                    k, static_cast<__nv_bfloat16*>(dx));
}

}  // namespace moe
