// Router: logits = x W_r (+ bias) in fp32 FMA, then per-token top-k and gates.
//
// The pages print no router; they cite the sparsely-gated MoE layer and Switch
// Transformers (FarSkip-Collective review, reference list) and name its cost
// T_gate in the overlap condition (ledger, Eq. 9).
//
// The logits must be fp32-accurate: routing is compared exactly with an fp64
// reference on inputs whose logit gaps are only 1e-4 of the logit scale.
//   bf16 layers: x is exactly bf16, and the fp32 router weight splits exactly
//     into three bf16 terms, W_r = W1 + W2 + W3 (8 + 8 + 8 significand bits; each
//     residual is exactly representable).  x . W_r = x.W1 + x.W2 + x.W3 with
//     every product exact and fp32 accumulation, i.e. fp32-accurate logits on the
//     tcgen05 tensor cores.  The three terms form one K range of 3d that is split
//     across CTAs; the top-k kernel adds the split partials in a fixed order.
//   fp32 layers: x is not bf16, so the logits run on the fp32 FMA pipe.
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
// Split K: CTA z of gridDim.z sums K range [z k_len, (z+1) k_len) and writes its
// partial logits at logits + z * T * E (k_len = d, one split, writes the logits).
template <typename TX, int BN>
__global__ void __launch_bounds__(kRThreads)
    router_logits_kernel(const TX* __restrict__ x, const float* __restrict__ W_r,
                         const float* __restrict__ bias, float* __restrict__ logits, int T, int d,
                         int E, int k_len) {
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
  const int k_begin = blockIdx.z * k_len;
  const int k_end = min(d, k_begin + k_len);
  logits += static_cast<long long>(blockIdx.z) * T * E;
  pdl_trigger();
  pdl_wait();
  for (int k0 = k_begin; k0 < k_end; k0 += kRBK) {
    {
      float v[4] = {0.f, 0.f, 0.f, 0.f};
      const int t = t0 + lm, kk = k0 + lk;
      if (t < T && kk < k_end) load4<TX>(x + static_cast<long long>(t) * d + kk, v);
#pragma unroll
      for (int i = 0; i < 4; ++i) xs[lk + i][lm] = v[i];
    }
    for (int i = tid; i < kRBK * BN; i += kRThreads) {
      const int kk = i / BN, n = i % BN;
      const int gk = k0 + kk, ge = e0 + n;
      ws[kk][n] = (gk < k_end && ge < E) ? W_r[static_cast<long long>(gk) * E + ge] : 0.f;
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

// W3[term][e][i] for term 0..2: W_r[i][e] = W3[0] + W3[1] + W3[2] exactly; rows e >= E are zero.
__global__ void __launch_bounds__(256)
    router_split_kernel(const float* __restrict__ W_r, int d, int E, int n_pad,
                        __nv_bfloat16* __restrict__ W3) {
  pdl_trigger();
  pdl_wait();
  const long long n = static_cast<long long>(n_pad) * d;
  for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < n;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int e = static_cast<int>(idx / d), i = static_cast<int>(idx - static_cast<long long>(e) * d);
    const float w = e < E ? W_r[static_cast<long long>(i) * E + e] : 0.f;
    const __nv_bfloat16 w1 = __float2bfloat16_rn(w);
    const float r1 = w - __bfloat162float(w1);
    const __nv_bfloat16 w2 = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(w2);
    W3[idx] = w1;
    W3[n + idx] = w2;
    W3[2 * n + idx] = __float2bfloat16_rn(r2);
  }
}

// Order-preserving 32-bit key of a logit: a larger logit has a larger key (-0 reads as +0 and
// NaN as -inf), and the key of any logit is above 0, the key of an empty slot.
__device__ __forceinline__ uint32_t logit_key(float v) {
  if (v != v) v = -INFINITY;
  if (v == 0.f) v = 0.f;
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_logit(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}
// compare-exchange for a descending sort of 64-bit keys
__device__ __forceinline__ void cas_desc(uint64_t& a, uint64_t& b) {
  const uint64_t hi = a > b ? a : b, lo = a > b ? b : a;
  a = hi;
  b = lo;
}

// One warp per token: logits = ordered sum of the split partials (+ bias), then the top k
// (ties -> lower expert), then gates.  Lane l holds experts l + 32 i, i < NV.  Each candidate
// is one 64-bit key, {logit key, 0xffff - expert}, so that the larger key is the better
// expert under the selection order; a lane sorts its NV keys, and each of the k rounds takes
// the warp's largest head (two warp max reductions: logit key, then expert among the equal
// logits) and pops it from its lane.
template <int NV>
__global__ void __launch_bounds__(256)
    router_topk_kernel(const float* __restrict__ part, int n_split, int ld,
                       const float* __restrict__ bias, float* __restrict__ logits_out,
                       int32_t* __restrict__ topk_idx, float* __restrict__ topk_gate, int T, int E,
                       int k, int gating) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  pdl_trigger();
  pdl_wait();
  if (warp >= T) return;
  // logits: the split partials added in split order.  Loads are issued kChunk
  // splits x NV expert slots at a time, so their latencies overlap.
  constexpr int kChunk = 4;
  float v[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? part[static_cast<long long>(warp) * ld + e] : 0.f;
  }
  for (int s0 = 1; s0 < n_split; s0 += kChunk) {
    float q[kChunk][NV];
#pragma unroll
    for (int u = 0; u < kChunk; ++u)
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int e = lane + 32 * i;
        q[u][i] = (e < E && s0 + u < n_split)
                      ? part[(static_cast<long long>(s0 + u) * T + warp) * ld + e]
                      : 0.f;
      }
#pragma unroll
    for (int u = 0; u < kChunk; ++u)
#pragma unroll
      for (int i = 0; i < NV; ++i)
        if (s0 + u < n_split) v[i] += q[u][i];
  }
  uint64_t key[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int e = lane + 32 * i;
    if (e < E) {
      if (bias) v[i] += bias[e];
      if (logits_out) logits_out[static_cast<long long>(warp) * E + e] = v[i];
      key[i] = (static_cast<uint64_t>(logit_key(v[i])) << 32) | static_cast<uint32_t>(0xffff - e);
    } else {
      v[i] = -INFINITY;
      key[i] = 0;
    }
  }
  // this lane's keys in descending order (sorting networks; e rises with i, so equal logits
  // keep the lower expert first)
  if (NV == 2) {
    cas_desc(key[0], key[1 % NV]);
  } else if (NV == 4) {
    cas_desc(key[0], key[1 % NV]); cas_desc(key[2 % NV], key[3 % NV]);
    cas_desc(key[0], key[2 % NV]); cas_desc(key[1 % NV], key[3 % NV]);
    cas_desc(key[1 % NV], key[2 % NV]);
  } else if (NV == 8) {
    cas_desc(key[0], key[1 % NV]); cas_desc(key[2 % NV], key[3 % NV]);
    cas_desc(key[4 % NV], key[5 % NV]); cas_desc(key[6 % NV], key[7 % NV]);
    cas_desc(key[0], key[2 % NV]); cas_desc(key[1 % NV], key[3 % NV]);
    cas_desc(key[4 % NV], key[6 % NV]); cas_desc(key[5 % NV], key[7 % NV]);
    cas_desc(key[1 % NV], key[2 % NV]); cas_desc(key[5 % NV], key[6 % NV]);
    cas_desc(key[0], key[4 % NV]); cas_desc(key[1 % NV], key[5 % NV]);
    cas_desc(key[2 % NV], key[6 % NV]); cas_desc(key[3 % NV], key[7 % NV]);
    cas_desc(key[2 % NV], key[4 % NV]); cas_desc(key[3 % NV], key[5 % NV]);
    cas_desc(key[1 % NV], key[2 % NV]); cas_desc(key[3 % NV], key[4 % NV]);
    cas_desc(key[5 % NV], key[6 % NV]);
  }
  // lane j < k keeps the j-th selection in registers
  float my_v = -INFINITY;
  int my_i = 0;
#pragma unroll 1
  for (int j = 0; j < k; ++j) {
    const uint32_t hh = static_cast<uint32_t>(key[0] >> 32);
    const uint32_t hl = static_cast<uint32_t>(key[0]);
    const uint32_t mh = __reduce_max_sync(0xffffffffu, hh);
    const uint32_t ml = __reduce_max_sync(0xffffffffu, hh == mh ? hl : 0u);
    if (hh == mh && hl == ml) {  // the lane holding the winner moves to its next key
#pragma unroll
      for (int i = 0; i + 1 < NV; ++i) key[i] = key[i + 1];
      key[NV - 1] = 0;
    }
    if (lane == j) {
      my_v = key_logit(mh);
      my_i = 0xffff - static_cast<int>(ml);
      if (mh == 0 || my_i < 0 || my_i >= E) my_i = 0;  // fewer than k experts: not reachable
    }
  }
  float g;
  if (gating == MOE_GATE_SIGMOID_TOPK) {
    g = 1.f / (1.f + expf(-my_v));
  } else {
    const float m = __shfl_sync(0xffffffffu, my_v, 0);  // the largest logit
    float z = 0.f;
    if (gating == MOE_GATE_SOFTMAX_TOPK) {
#pragma unroll
      for (int i = 0; i < NV; ++i) z += (lane + 32 * i < E) ? expf(v[i] - m) : 0.f;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
    } else {
      // the selected terms added in selection order
      const float t = lane < k ? expf(my_v - m) : 0.f;
      for (int j = 0; j < k; ++j) z += __shfl_sync(0xffffffffu, t, j);
    }
    g = expf(my_v - m) / z;
  }
  if (lane < k) {
    topk_idx[static_cast<long long>(warp) * k + lane] = my_i;
    topk_gate[static_cast<long long>(warp) * k + lane] = g;
  }
}

template <typename TX>
cudaError_t logits_dispatch(const TX* x, const float* W_r, const float* bias, float* logits, int T,
                            int d, int E, int n_split, cudaStream_t s) {
  const int gx = ceil_div(T, kRBM);
  const int k_len = d / n_split;
  if (E <= 16)
    return launch_pdl(router_logits_kernel<TX, 16>, dim3(gx, 1, n_split), dim3(kRThreads), 0, s,
                      x, W_r, bias, logits, T, d, E, k_len);
  if (E <= 32)
    return launch_pdl(router_logits_kernel<TX, 32>, dim3(gx, 1, n_split), dim3(kRThreads), 0, s,
                      x, W_r, bias, logits, T, d, E, k_len);
  return launch_pdl(router_logits_kernel<TX, 64>, dim3(gx, ceil_div(E, 64), n_split),
                    dim3(kRThreads), 0, s, x, W_r, bias, logits, T, d, E, k_len);
}

}  // namespace

cudaError_t launch_router_logits(int act_dtype, const void* x, const float* W_r, const float* bias,
                                 float* logits, int T, int d, int E, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  if (act_dtype == MOE_F32)
    return logits_dispatch(static_cast<const float*>(x), W_r, bias, logits, T, d, E, 1, stream);
  return logits_dispatch(static_cast<const __nv_bfloat16*>(x), W_r, bias, logits, T, d, E, 1,
                         stream);
}

cudaError_t launch_router_topk(const float* part, int n_split, int ld, const float* bias,
                               float* logits_out, int32_t* topk_idx, float* topk_gate, int T,
                               int E, int k, int gating, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const int warps_per_block = 8;
  const dim3 grid(ceil_div(T, warps_per_block)), block(32 * warps_per_block);
  if (E <= 32)
    return launch_pdl(router_topk_kernel<1>, grid, block, 0, stream, part, n_split, ld, bias,
                      logits_out, topk_idx, topk_gate, T, E, k, gating);
  if (E <= 64)
    return launch_pdl(router_topk_kernel<2>, grid, block, 0, stream, part, n_split, ld, bias,
                      logits_out, topk_idx, topk_gate, T, E, k, gating);
  if (E <= 128)
    return launch_pdl(router_topk_kernel<4>, grid, block, 0, stream, part, n_split, ld, bias,
                      logits_out, topk_idx, topk_gate, T, E, k, gating);
  return launch_pdl(router_topk_kernel<8>, grid, block, 0, stream, part, n_split, ld, bias,
                    logits_out, topk_idx, topk_gate, T, E, k, gating);
}

int router_n_pad(int E) { return ceil_div(E, 32) * 32; }

// The three terms sit side by side along N: in one MMA up to 64 experts (N = 3 x E rounded up
// to 32, at most 256), in two (terms 1 and 2, then term 3) up to 128.
static bool router_stacked(int E) { return 3 * router_n_pad(E) <= 384; }

// K splits: the largest divisor of the K blocks (d/64 with the terms side by side, else
// 3d/64) that keeps the tile count (m-tiles x splits) within one wave of CTAs, and at most
// 8, so that the top-k kernel adds few partials (a batch of a few m-tiles would otherwise
// take one split per K block).
int router_splits(int T, int d, int E, int num_sms) {
  const int kb = (router_stacked(E) ? 1 : 3) * (d / kTcTileK);
  const int mtiles = ceil_div(T, kMTile);
  const int target = max(1, min(8, num_sms / max(1, mtiles)));
  int best = 1;
  for (int s = 1; s <= min(kb, target); ++s)
    if (kb % s == 0) best = s;
  return best;
}

size_t router_scratch_bytes(int T, int d, int E, int num_sms) {
  const size_t n_pad = router_n_pad(E);
  const size_t w3 = (3 * n_pad * d * sizeof(__nv_bfloat16) + 255) & ~size_t(255);
  const size_t part =
      static_cast<size_t>(router_splits(T, d, E, num_sms)) * T * n_pad * sizeof(float);
  return w3 + part;
}

cudaError_t launch_router_tc(const void* x, const float* W_r, int T, int d, int E, int num_sms,
                             void* scratch, const float** part_out, int* n_split, int* ld,
                             unsigned* status, cudaStream_t stream) {
  const int n_pad = router_n_pad(E);
  const int splits = router_splits(T, d, E, num_sms);
  const bool stacked = router_stacked(E);
  __nv_bfloat16* W3 = static_cast<__nv_bfloat16*>(scratch);
  float* part = reinterpret_cast<float*>(static_cast<char*>(scratch) +
                                         ((3 * static_cast<size_t>(n_pad) * d * 2 + 255) & ~size_t(255)));
  const long long n = static_cast<long long>(n_pad) * d;
  const int split_blocks = static_cast<int>(n / 256 + 1 < 2048 ? n / 256 + 1 : 2048);
  cudaError_t err = launch_pdl(router_split_kernel, dim3(split_blocks), dim3(256), 0, stream, W_r,
                               d, E, n_pad, W3);
  if (err != cudaSuccess) return err;
  TcGemmArgs a = {};
  a.n_ntiles = splits;
  a.n_kblocks = (stacked ? 1 : 3) * (d / kTcTileK) / splits;
  a.router_stacked = stacked ? 1 : 0;
  a.kb_per_slice = a.n_kblocks;
  a.nt_per_slice = splits;
  a.router_n = n_pad;
  a.router_kbd = d / kTcTileK;
  a.n_rows = T;
  a.part = part;
  a.status = status;
  const int tiles = ceil_div(T, kMTile) * splits;
  err = tc_gemm(kTcRouter, x, T, d, W3, 3, n_pad, d, a, min(num_sms, tiles), stream);
  *part_out = part;
  *n_split = splits;
  *ld = n_pad;
  return err;
}

}  // namespace moe
