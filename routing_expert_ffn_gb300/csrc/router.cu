// Router: logits = x W_r (+ bias) in fp32 FMA, then per-token top-k and gates.
//
// The pages print no router; they cite the sparsely-gated MoE layer and Switch
// Transformers (FarSkip-Collective review, reference list) and name its cost
// T_gate in the overlap condition (ledger, Eq. 9).  The logits are an fp32
// contraction with E <= 256 columns: too narrow and too precision-sensitive for
// the bf16 tensor path (routing must agree bit for bit with an fp64 reference
// on inputs with relative logit gaps of 1e-4), so it runs on the fp32 pipe.
#include <float.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kRBM = 64;   // tokens per CTA
constexpr int kRBK = 16;   // K per smem stage
constexpr int kRThreads = 256;

template <typename TX>
__device__ __forceinline__ void load4(const TX* p, float* v);
template <>
__device__ __forceinline__ void load4<float>(const float* p, float* v) {
  float4 a = *reinterpret_cast<const float4*>(p);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
}
template <>
__device__ __forceinline__ void load4<__nv_bfloat16>(const __nv_bfloat16* p, float* v) {
  uint2 a = *reinterpret_cast<const uint2*>(p);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&a);
  float2 f0 = __bfloat1622float2(h[0]), f1 = __bfloat1622float2(h[1]);
  v[0] = f0.x; v[1] = f0.y; v[2] = f1.x; v[3] = f1.y;
}

// CTA tile: 64 tokens x BN experts; thread tile TM tokens x 4 experts, TM = BN / 16.
template <typename TX, int BN>
__global__ void __launch_bounds__(kRThreads)
    router_logits_kernel(const TX* __restrict__ x, const float* __restrict__ W_r,
                         const float* __restrict__ bias, float* __restrict__ logits, int T, int d,
                         int E) {
  constexpr int TM = BN / 16;
  constexpr int NX = BN / 4;  // threads along experts
  __shared__ __align__(16) float xs[kRBK][kRBM + 4];
  __shared__ __align__(16) float ws[kRBK][BN];
  const int tid = threadIdx.x;
  const int tx = tid % NX, ty = tid / NX;
  const int t0 = blockIdx.x * kRBM;
  const int e0 = blockIdx.y * BN;
  float acc[TM][4];
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

  // x tile loader: 64 rows x 16 k = 256 threads x 4 consecutive k
  const int lm = tid >> 2, lk = (tid & 3) * 4;
  for (int k0 = 0; k0 < d; k0 += kRBK) {
    {
      float v[4] = {0.f, 0.f, 0.f, 0.f};
      const int t = t0 + lm, kk = k0 + lk;
      if (t < T && kk < d) load4<TX>(x + static_cast<long long>(t) * d + kk, v);
#pragma unroll
      for (int i = 0; i < 4; ++i) xs[lk + i][lm] = v[i];
    }
    for (int i = tid; i < kRBK * BN; i += kRThreads) {
      const int kk = i / BN, n = i % BN;
      const int gk = k0 + kk, ge = e0 + n;
      ws[kk][n] = (gk < d && ge < E) ? W_r[static_cast<long long>(gk) * E + ge] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kRBK; ++kk) {
      float a[TM];
#pragma unroll
      for (int i = 0; i < TM; ++i) a[i] = xs[kk][ty * TM + i];
      const float4 b = *reinterpret_cast<const float4*>(&ws[kk][tx * 4]);
#pragma unroll
      for (int i = 0; i < TM; ++i) {
        acc[i][0] = fmaf(a[i], b.x, acc[i][0]);
        acc[i][1] = fmaf(a[i], b.y, acc[i][1]);
        acc[i][2] = fmaf(a[i], b.z, acc[i][2]);
        acc[i][3] = fmaf(a[i], b.w, acc[i][3]);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < TM; ++i) {
    const int t = t0 + ty * TM + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + tx * 4 + j;
      if (e < E) logits[static_cast<long long>(t) * E + e] = acc[i][j] + (bias ? bias[e] : 0.f);
    }
  }
}

// One warp per token: k rounds of warp argmax (ties -> lower expert), then gates.
__global__ void __launch_bounds__(256)
    router_topk_kernel(const float* __restrict__ logits, int32_t* __restrict__ topk_idx,
                       float* __restrict__ topk_gate, int T, int E, int k, int gating) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= T) return;
  const float* row = logits + static_cast<long long>(warp) * E;
  float v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? row[e] : -INFINITY;
  }
  unsigned taken = 0;
  float sel_v[32];
  int sel_i[32];
#pragma unroll 1
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((taken >> i) & 1u) && (v[i] > bv || (v[i] == bv && e < bi))) {
        bv = v[i];
        bi = e;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (bi >= E) bi = 0;  // only reachable with NaN logits
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    sel_v[j] = bv;
    sel_i[j] = bi;
  }
  float g[32];
  if (gating == MOE_GATE_SIGMOID_TOPK) {
    for (int j = 0; j < k; ++j) g[j] = 1.f / (1.f + expf(-sel_v[j]));
  } else {
    const float m = sel_v[0];
    float z = 0.f;
    if (gating == MOE_GATE_SOFTMAX_TOPK) {
#pragma unroll
      for (int i = 0; i < 8; ++i) z += (lane + 32 * i < E) ? expf(v[i] - m) : 0.f;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
    } else {
      for (int j = 0; j < k; ++j) z += expf(sel_v[j] - m);
    }
    for (int j = 0; j < k; ++j) g[j] = expf(sel_v[j] - m) / z;
  }
  for (int j = lane; j < k; j += 32) {
    topk_idx[static_cast<long long>(warp) * k + j] = sel_i[j];
    topk_gate[static_cast<long long>(warp) * k + j] = g[j];
  }
}

template <typename TX>
cudaError_t logits_dispatch(const TX* x, const float* W_r, const float* bias, float* logits, int T,
                            int d, int E, cudaStream_t s) {
  const int gx = ceil_div(T, kRBM);
  if (E <= 16) {
    router_logits_kernel<TX, 16><<<dim3(gx, 1), kRThreads, 0, s>>>(x, W_r, bias, logits, T, d, E);
  } else if (E <= 32) {
    router_logits_kernel<TX, 32><<<dim3(gx, 1), kRThreads, 0, s>>>(x, W_r, bias, logits, T, d, E);
  } else {
    router_logits_kernel<TX, 64>
        <<<dim3(gx, ceil_div(E, 64)), kRThreads, 0, s>>>(x, W_r, bias, logits, T, d, E);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_router_logits(int act_dtype, const void* x, const float* W_r, const float* bias,
                                 float* logits, int T, int d, int E, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  if (act_dtype == MOE_F32)
    return logits_dispatch(static_cast<const float*>(x), W_r, bias, logits, T, d, E, stream);
  return logits_dispatch(static_cast<const __nv_bfloat16*>(x), W_r, bias, logits, T, d, E,
                         stream);
}

cudaError_t launch_router_topk(const float* logits, int32_t* topk_idx, float* topk_gate, int T,
                               int E, int k, int gating, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const int warps_per_block = 8;
  router_topk_kernel<<<ceil_div(T, warps_per_block), 32 * warps_per_block, 0, stream>>>(
      logits, topk_idx, topk_gate, T, E, k, gating);
  return cudaGetLastError();
}

}  // namespace moe
