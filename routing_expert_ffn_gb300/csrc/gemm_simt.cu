// fp32 grouped GEMM on the FMA pipe, for fp32 layers (the tensor cores' TF32
// mode would miss a 1e-4 relative tolerance).  Same m-tile tables and slice
// conventions as the tcgen05 path:
//   swiglu: h[row, nt*64 + n] = SiLU(A[row] . Bg[n]) * (A[row] . Bu[n]) over a
//           64-hidden-unit tile whose gate rows are n0.. and up rows up_off+n0..
//   store:  out[map(row), nt*64 + n] = sum_k A[row, k] * B[slice(k), n, k mod k_per_slice]
// CTA: one 128-row m-tile x 64 output columns, 256 threads, 8x4 per thread.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int SBM = 128, SBN = 64, SBK = 16;

__device__ __forceinline__ void load_tile_rows(float (*dst)[SBM + 4], const float* src,
                                               long long ld, int row_limit, int k0, int K,
                                               const int* row_index /* 128 source rows */) {
  // 128 rows x 16 k = 512 float4; 256 threads x 2
  for (int i = threadIdx.x; i < SBM * SBK / 4; i += blockDim.x) {
    const int r = i >> 2, kq = (i & 3) * 4;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    const int sr = row_index[r];
    if (sr >= 0 && r < row_limit && k0 + kq < K)
      v = *reinterpret_cast<const float4*>(src + sr * ld + k0 + kq);
    dst[kq + 0][r] = v.x;
    dst[kq + 1][r] = v.y;
    dst[kq + 2][r] = v.z;
    dst[kq + 3][r] = v.w;
  }
}

template <bool SWIGLU>
__global__ void __launch_bounds__(256)
    simt_gemm_kernel(const float* __restrict__ A, const float* __restrict__ B, int b_rows,
                     int K_total, int k_per_slice, int nt_per_slice, int b_up_offset,
                     const int4* __restrict__ mt_info, const int32_t* __restrict__ group_mt_begin,
                     int n_groups, const int32_t* __restrict__ out_rowmap, float* __restrict__ out,
                     long long ld_out) {
  __shared__ __align__(16) float As[SBK][SBM + 4];
  __shared__ __align__(16) float Bs[SBK][SBM + 4];  // SWIGLU: 64 gate + 64 up columns
  __shared__ int a_rows[SBM];
  __shared__ int b_rows_idx[SBM];
  const int mt = blockIdx.y;
  if (mt >= group_mt_begin[n_groups]) return;
  const int4 m = mt_info[mt];
  const int nt = blockIdx.x;
  const int nslice = nt / nt_per_slice;
  const int n0 = (nt - nslice * nt_per_slice) * SBN;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int nb = SWIGLU ? 2 * SBN : SBN;
  float acc[8][4], acc2[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = acc2[i][j] = 0.f;

  for (int i = threadIdx.x; i < SBM; i += blockDim.x) a_rows[i] = i < m.z ? m.y + i : -1;
  for (int k0 = 0; k0 < K_total; k0 += SBK) {
    const int kslice = SWIGLU ? 0 : k0 / k_per_slice;
    const int kin = k0 - kslice * k_per_slice;
    const int slice = m.x + nslice + kslice;
    const float* Bs_base = B + static_cast<long long>(slice) * b_rows * k_per_slice;
    __syncthreads();
    for (int i = threadIdx.x; i < SBM; i += blockDim.x) {
      int r = -1;
      if (i < nb) r = SWIGLU ? (i < SBN ? n0 + i : b_up_offset + n0 + i - SBN) : n0 + i;
      b_rows_idx[i] = r;
    }
    __syncthreads();
    load_tile_rows(As, A, K_total, SBM, k0, K_total, a_rows);
    load_tile_rows(Bs, Bs_base, k_per_slice, nb, kin, k_per_slice, b_rows_idx);
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < SBK; ++kk) {
      const float4 a0 = *reinterpret_cast<const float4*>(&As[kk][ty * 8]);
      const float4 a1 = *reinterpret_cast<const float4*>(&As[kk][ty * 8 + 4]);
      const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float4 b = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        acc[i][0] = fmaf(a[i], b.x, acc[i][0]);
        acc[i][1] = fmaf(a[i], b.y, acc[i][1]);
        acc[i][2] = fmaf(a[i], b.z, acc[i][2]);
        acc[i][3] = fmaf(a[i], b.w, acc[i][3]);
      }
      if (SWIGLU) {
        const float4 u = *reinterpret_cast<const float4*>(&Bs[kk][SBN + tx * 4]);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          acc2[i][0] = fmaf(a[i], u.x, acc2[i][0]);
          acc2[i][1] = fmaf(a[i], u.y, acc2[i][1]);
          acc2[i][2] = fmaf(a[i], u.z, acc2[i][2]);
          acc2[i][3] = fmaf(a[i], u.w, acc2[i][3]);
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = ty * 8 + i;
    if (r >= m.z) continue;
    long long orow = m.y + r;
    if (!SWIGLU && out_rowmap) orow = out_rowmap[orow];
    float v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (SWIGLU) {
        const float g = acc[i][j];
        v[j] = g / (1.f + expf(-g)) * acc2[i][j];
      } else {
        v[j] = acc[i][j];
      }
    }
    *reinterpret_cast<float4*>(out + orow * ld_out + static_cast<long long>(nt) * SBN + tx * 4) =
        make_float4(v[0], v[1], v[2], v[3]);
  }
}

}  // namespace

cudaError_t simt_gemm_swiglu(const float* A, const float* B, int b_slices, int b_rows, int K,
                             int kb_per_slice_k, int nt_per_slice, int H_total, int b_up_offset,
                             const int4* mt_info, const int32_t* group_mt_begin, int n_groups,
                             int max_mt, float* out, cudaStream_t stream) {
  (void)b_slices;
  (void)kb_per_slice_k;
  if (max_mt <= 0) return cudaSuccess;
  dim3 grid(H_total / SBN, max_mt);
  simt_gemm_kernel<true><<<grid, 256, 0, stream>>>(A, B, b_rows, K, K, nt_per_slice / 1,
                                                    b_up_offset, mt_info, group_mt_begin, n_groups,
                                                    nullptr, out, H_total);
  return cudaGetLastError();
}

cudaError_t simt_gemm_store(const float* A, const float* B, int b_slices, int b_rows, int K,
                            int k_per_slice, int N, const int4* mt_info,
                            const int32_t* group_mt_begin, int n_groups, int max_mt,
                            const int32_t* out_rowmap, float* out, cudaStream_t stream) {
  (void)b_slices;
  if (max_mt <= 0) return cudaSuccess;
  dim3 grid(N / SBN, max_mt);
  simt_gemm_kernel<false><<<grid, 256, 0, stream>>>(A, B, b_rows, K, k_per_slice, N / SBN, 0,
                                                     mt_info, group_mt_begin, n_groups, out_rowmap,
                                                     out, N);
  return cudaGetLastError();
}

}  // namespace moe
